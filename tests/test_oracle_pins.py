"""Pins for the CPU oracle: each check comes from something other than the oracle.

* hand-derived worked examples (tests/golden/);
* a brute-force dense-mask statement of the per-document causal rule of
  cp_blockdiag_sdpa (page "nemo_automodel.components.distributed.blockdiag_cp"),
  written with pure-Python loops and math.exp;
* torch's own scaled_dot_product_attention (CPU, fp64, is_causal) for the
  special case of one document, forward and autograd backward;
* closed forms (q = 0, length-1 documents), invariants (padding, GQA, query
  intervals, id renumbering) and central finite differences of the forward.
"""
import math
import os

import numpy as np
import pytest
import torch

from oracle import blockdiag as orc

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_rows(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append([int(x) for x in line.split()])
    return rows


# ---------------------------------------------------------------- ids / segments

def test_golden_tiny_doc_ids():
    runs = _read_rows("tiny_doc_ids.txt")
    expect = np.concatenate([np.full(n, i, np.int32) for i, n in runs])
    ids = orc.doc_ids_from_cu_seqlens([0, 37, 137, 138, 202, 256], 256)
    assert ids.dtype == np.int32
    np.testing.assert_array_equal(ids, expect)


def test_golden_tiny_segments():
    bounds, sids = _read_rows("tiny_segments.txt")
    ids = orc.doc_ids_from_cu_seqlens([0, 37, 137, 138, 202, 256], 256)
    seg, seg_ids = orc.segment_cu_seqlens(ids)
    np.testing.assert_array_equal(seg, bounds)
    np.testing.assert_array_equal(seg_ids, sids)


def test_golden_padded_small():
    cu, (S,), ids_expect, seg_expect, sid_expect = _read_rows("padded_small.txt")
    ids = orc.doc_ids_from_cu_seqlens(cu, S)
    np.testing.assert_array_equal(ids, ids_expect)
    seg, sid = orc.segment_cu_seqlens(ids)
    np.testing.assert_array_equal(seg, seg_expect)
    np.testing.assert_array_equal(sid, sid_expect)


@pytest.mark.parametrize("seed", range(20))
def test_doc_ids_properties(seed):
    rng = np.random.default_rng(seed)
    S = int(rng.integers(1, 300))
    n = int(rng.integers(1, 9))
    cu = np.concatenate([[0], np.sort(rng.integers(0, S + 1, n))]).astype(np.int32)
    ids = orc.doc_ids_from_cu_seqlens(cu, S)
    assert ids.shape == (S,)
    for d in range(n):  # each document's positions carry d+1, count = its length
        assert np.count_nonzero(ids == d + 1) == cu[d + 1] - cu[d]
    assert np.count_nonzero(ids == 0) == S - cu[-1]
    assert np.all(ids[cu[-1]:] == 0)
    seg, sid = orc.segment_cu_seqlens(ids)
    assert seg[0] == 0 and seg[-1] == S and np.all(np.diff(seg) > 0)
    for a in range(sid.size):  # runs are constant and maximal
        assert np.all(ids[seg[a]:seg[a + 1]] == sid[a])
        if a > 0:
            assert sid[a] != sid[a - 1]


@pytest.mark.parametrize("bad", [[1, 4], [0, 5, 3], [0, 9]])
def test_doc_ids_rejects_invalid(bad):
    with pytest.raises(ValueError):
        orc.doc_ids_from_cu_seqlens(bad, 8)


def test_segments_split_repeated_ids():
    ids = np.array([1, 1, 2, 2, 1, 1, 0, 0], np.int32)
    seg, sid = orc.segment_cu_seqlens(ids)
    np.testing.assert_array_equal(seg, [0, 2, 4, 6, 8])
    np.testing.assert_array_equal(sid, [1, 2, 1, 0])


# ---------------------------------------------------------------- brute force

def _brute_forward(q, k, v, ids, seq_start, scale, G):
    """Dense mask from the rule, written element by element."""
    B, Hq, L, D = q.shape
    S = k.shape[2]
    out = np.zeros((B, Hq, L, D))
    lse = np.full((B, Hq, L), -math.inf)
    for b in range(B):
        for h in range(Hq):
            g = h // G
            for i in range(L):
                t = seq_start + i
                if ids[b][t] == 0:
                    continue
                allowed = [j for j in range(S)
                           if j <= t and all(ids[b][x] == ids[b][t] for x in range(j, t + 1))]
                s = {j: scale * sum(float(q[b, h, i, d]) * float(k[b, g, j, d]) for d in range(D))
                     for j in allowed}
                z = sum(math.exp(x) for x in s.values())
                lse[b, h, i] = math.log(z)
                for j in allowed:
                    w = math.exp(s[j]) / z
                    for d in range(D):
                        out[b, h, i, d] += w * float(v[b, g, j, d])
    return out, lse


def _rand(shape, rng):
    return rng.standard_normal(shape)


@pytest.mark.parametrize("case", [
    # (ids row(s), seq_start, L, Hq, Hkv, D)
    ([[1, 1, 1, 2, 2, 3, 3, 3, 3, 0, 0]], 0, 11, 2, 1, 3),
    ([[1, 1, 2, 2, 1, 1, 0, 0]], 0, 8, 2, 2, 4),           # repeated id, split runs
    ([[4, 4, 4, 4, 4, 7, 7, 7, 0, 0, 9, 9]], 3, 6, 4, 2, 2),  # interval, interior pad
    ([[1] * 9, [2, 2, 0, 3, 3, 3, 3, 3, 3]], 2, 5, 2, 1, 3),  # two rows
])
def test_forward_matches_brute_force(case):
    rows, seq_start, L, Hq, Hkv, D = case
    rng = np.random.default_rng(7)
    ids = np.asarray(rows, np.int32)
    B, S = ids.shape
    q = _rand((B, Hq, L, D), rng)
    k = _rand((B, Hkv, S, D), rng)
    v = _rand((B, Hkv, S, D), rng)
    scale = D ** -0.5
    out, lse = orc.blockdiag_sdpa_forward(q, k, v, ids, seq_start, None, Hq != Hkv)
    bo, bl = _brute_forward(q, k, v, ids, seq_start, scale, Hq // Hkv)
    np.testing.assert_allclose(out, bo, rtol=1e-12, atol=1e-12)
    np.testing.assert_array_equal(np.isinf(lse), np.isinf(bl))
    fin = np.isfinite(bl)
    np.testing.assert_allclose(lse[fin], bl[fin], rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- torch SDPA special case

def _torch_causal(q, k, v, scale):
    """torch SDPA, fp64 CPU, one causal document; returns out and grads vs dO."""
    tq, tk, tv = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (q, k, v))
    o = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=True, scale=scale)
    return tq, tk, tv, o


@pytest.mark.parametrize("D", [8, 16])
def test_single_document_is_torch_causal_sdpa(D):
    rng = np.random.default_rng(D)
    S, H = 37, 2
    q, k, v, do = (_rand((1, H, S, D), rng) for _ in range(4))
    ids = np.ones((1, S), np.int32)
    out, lse = orc.blockdiag_sdpa_forward(q, k, v, ids)
    dq, dk, dv = orc.blockdiag_sdpa_backward(q, k, v, do, ids)
    tq, tk, tv, o = _torch_causal(q, k, v, D ** -0.5)
    o.backward(torch.tensor(do))
    np.testing.assert_allclose(out, o.detach().numpy(), rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(dq, tq.grad.numpy(), rtol=1e-10, atol=1e-11)
    np.testing.assert_allclose(dk, tk.grad.numpy(), rtol=1e-10, atol=1e-11)
    np.testing.assert_allclose(dv, tv.grad.numpy(), rtol=1e-10, atol=1e-11)
    # lse against a logsumexp of the torch-visible scores
    s = torch.tensor(q[0]) @ torch.tensor(k[0]).transpose(-1, -2) * D ** -0.5
    s = s.masked_fill(torch.ones(S, S, dtype=torch.bool).triu(1), -math.inf)
    np.testing.assert_allclose(lse[0], torch.logsumexp(s, -1).numpy(), rtol=1e-12, atol=1e-12)


def test_packed_equals_documents_run_separately():
    """Block-diagonal result = each document alone through torch causal SDPA."""
    rng = np.random.default_rng(3)
    cu = [0, 5, 17, 18, 40, 52]
    S, Hq, Hkv, D = 60, 4, 2, 8
    ids = orc.doc_ids_from_cu_seqlens(cu, S)[None]
    q, do = _rand((1, Hq, S, D), rng), _rand((1, Hq, S, D), rng)
    k, v = _rand((1, Hkv, S, D), rng), _rand((1, Hkv, S, D), rng)
    out, _ = orc.blockdiag_sdpa_forward(q, k, v, ids, enable_gqa=True)
    dq, dk, dv = orc.blockdiag_sdpa_backward(q, k, v, do, ids, enable_gqa=True)
    e_out, e_dq = np.zeros_like(out), np.zeros_like(dq)
    e_dk, e_dv = np.zeros_like(dk), np.zeros_like(dv)
    for a, b in zip(cu[:-1], cu[1:]):
        if a == b:
            continue
        kk = np.repeat(k[:, :, a:b], 2, axis=1)
        vv = np.repeat(v[:, :, a:b], 2, axis=1)
        tq, tk, tv, o = _torch_causal(q[:, :, a:b], kk, vv, D ** -0.5)
        o.backward(torch.tensor(do[:, :, a:b]))
        e_out[:, :, a:b] = o.detach().numpy()
        e_dq[:, :, a:b] = tq.grad.numpy()
        e_dk[:, :, a:b] = tk.grad.numpy().reshape(1, Hkv, 2, b - a, D).sum(2)
        e_dv[:, :, a:b] = tv.grad.numpy().reshape(1, Hkv, 2, b - a, D).sum(2)
    for got, exp in ((out, e_out), (dq, e_dq), (dk, e_dk), (dv, e_dv)):
        np.testing.assert_allclose(got, exp, rtol=1e-10, atol=1e-11)
    # padding rows: output 0, keys past the last document receive no gradient
    assert np.all(out[:, :, 52:] == 0) and np.all(dq[:, :, 52:] == 0)
    assert np.all(dk[:, :, 52:] == 0) and np.all(dv[:, :, 52:] == 0)


# ---------------------------------------------------------------- closed forms

def test_length_one_documents_return_v():
    rng = np.random.default_rng(11)
    S, D = 9, 4
    cu = list(range(S + 1))  # every document has one token
    ids = orc.doc_ids_from_cu_seqlens(cu, S)[None]
    q, k, v = (_rand((1, 1, S, D), rng) for _ in range(3))
    out, lse = orc.blockdiag_sdpa_forward(q, k, v, ids)
    np.testing.assert_array_equal(out, v)
    np.testing.assert_allclose(lse[0, 0], D ** -0.5 * (q[0, 0] * k[0, 0]).sum(-1), rtol=1e-14)


def test_zero_queries_closed_form():
    """q = 0: uniform weights over the document prefix."""
    rng = np.random.default_rng(5)
    cu, S, D = [0, 6, 13, 20], 24, 3
    ids = orc.doc_ids_from_cu_seqlens(cu, S)[None]
    q = np.zeros((1, 1, S, D))
    k, v, do = (_rand((1, 1, S, D), rng) for _ in range(3))
    out, lse = orc.blockdiag_sdpa_forward(q, k, v, ids)
    _, _, dv = orc.blockdiag_sdpa_backward(q, k, v, do, ids)
    for a, b in zip(cu[:-1], cu[1:]):
        for t in range(a, b):
            n = t - a + 1
            assert lse[0, 0, t] == pytest.approx(math.log(n), abs=1e-14)
            np.testing.assert_allclose(out[0, 0, t], v[0, 0, a:t + 1].mean(0), rtol=1e-13)
        for j in range(a, b):  # dv_j = sum_{i >= j} dO_i / (i - a + 1)
            e = sum(do[0, 0, i] / (i - a + 1) for i in range(j, b))
            np.testing.assert_allclose(dv[0, 0, j], e, rtol=1e-12, atol=1e-14)
    assert np.all(np.isneginf(lse[0, 0, 20:]))


# ---------------------------------------------------------------- invariants

def test_gqa_equals_mha_on_repeated_kv():
    rng = np.random.default_rng(9)
    S, Hq, Hkv, D = 30, 6, 2, 4
    ids = orc.doc_ids_from_cu_seqlens([0, 11, 25], S)[None]
    q, do = _rand((1, Hq, S, D), rng), _rand((1, Hq, S, D), rng)
    k, v = _rand((1, Hkv, S, D), rng), _rand((1, Hkv, S, D), rng)
    o1, l1 = orc.blockdiag_sdpa_forward(q, k, v, ids, enable_gqa=True)
    g1 = orc.blockdiag_sdpa_backward(q, k, v, do, ids, enable_gqa=True)
    kr, vr = np.repeat(k, 3, axis=1), np.repeat(v, 3, axis=1)
    o2, l2 = orc.blockdiag_sdpa_forward(q, kr, vr, ids)
    g2 = orc.blockdiag_sdpa_backward(q, kr, vr, do, ids)
    np.testing.assert_allclose(o1, o2, rtol=1e-13, atol=1e-14)
    np.testing.assert_array_equal(l1, l2)
    np.testing.assert_allclose(g1[0], g2[0], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(g1[1], g2[1].reshape(1, 2, 3, S, D).sum(2), rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(g1[2], g2[2].reshape(1, 2, 3, S, D).sum(2), rtol=1e-12, atol=1e-13)
    with pytest.raises(ValueError):
        orc.blockdiag_sdpa_forward(q, k, v, ids, enable_gqa=False)


def test_intervals_concatenate_to_full_rows():
    """Queries split into contiguous intervals against the full K/V row."""
    rng = np.random.default_rng(13)
    S, L, Hq, Hkv, D = 48, 12, 2, 1, 4
    ids = orc.doc_ids_from_cu_seqlens([0, 7, 30, 31, 45], S)[None]
    q, do = _rand((1, Hq, S, D), rng), _rand((1, Hq, S, D), rng)
    k, v = _rand((1, Hkv, S, D), rng), _rand((1, Hkv, S, D), rng)
    out, lse = orc.blockdiag_sdpa_forward(q, k, v, ids, enable_gqa=True)
    dq, dk, dv = orc.blockdiag_sdpa_backward(q, k, v, do, ids, enable_gqa=True)
    sk, sv = np.zeros_like(dk), np.zeros_like(dv)
    for s0 in range(0, S, L):
        o_i, l_i = orc.blockdiag_sdpa_forward(q[:, :, s0:s0 + L], k, v, ids, s0, None, True)
        g = orc.blockdiag_sdpa_backward(q[:, :, s0:s0 + L], k, v, do[:, :, s0:s0 + L], ids, s0,
                                        None, True)
        np.testing.assert_allclose(o_i, out[:, :, s0:s0 + L], rtol=1e-13, atol=1e-14)
        np.testing.assert_allclose(l_i, lse[:, :, s0:s0 + L], rtol=1e-13, atol=1e-14)
        np.testing.assert_allclose(g[0], dq[:, :, s0:s0 + L], rtol=1e-12, atol=1e-13)
        assert np.all(g[1][:, :, s0 + L:] == 0) and np.all(g[2][:, :, s0 + L:] == 0)
        sk += g[1]
        sv += g[2]
    np.testing.assert_allclose(sk, dk, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(sv, dv, rtol=1e-12, atol=1e-13)


def test_renumbering_ids_changes_nothing():
    rng = np.random.default_rng(17)
    S, D = 20, 4
    a = np.array([1] * 6 + [2] * 5 + [3] * 6 + [0] * 3, np.int32)[None]
    b = np.array([8] * 6 + [5] * 5 + [8] * 6 + [0] * 3, np.int32)[None]
    q, k, v, do = (_rand((1, 2, S, D), rng) for _ in range(4))
    oa, la = orc.blockdiag_sdpa_forward(q, k, v, a)
    ob, lb = orc.blockdiag_sdpa_forward(q, k, v, b)
    np.testing.assert_array_equal(oa, ob)
    np.testing.assert_array_equal(la, lb)
    ga = orc.blockdiag_sdpa_backward(q, k, v, do, a)
    gb = orc.blockdiag_sdpa_backward(q, k, v, do, b)
    for x, y in zip(ga, gb):
        np.testing.assert_array_equal(x, y)


def test_probabilities_sum_to_one_and_scale_default():
    """sum_j p_ij = 1: a constant v gives a constant o; scale None means D**-0.5."""
    rng = np.random.default_rng(19)
    S, D = 25, 8
    ids = orc.doc_ids_from_cu_seqlens([0, 10, 25], S)[None]
    q, k = _rand((1, 1, S, D), rng), _rand((1, 1, S, D), rng)
    out, _ = orc.blockdiag_sdpa_forward(q, k, np.full((1, 1, S, D), 3.25), ids)
    np.testing.assert_allclose(out, 3.25, rtol=1e-14)
    v = _rand((1, 1, S, D), rng)
    o1, l1 = orc.blockdiag_sdpa_forward(q, k, v, ids, scale=None)
    o2, l2 = orc.blockdiag_sdpa_forward(q, k, v, ids, scale=D ** -0.5)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)
    _, l3 = orc.blockdiag_sdpa_forward(q, k, v, ids, scale=0.5)
    assert not np.allclose(l1, l3)


# ---------------------------------------------------------------- finite differences

def test_backward_matches_finite_differences():
    rng = np.random.default_rng(23)
    S, L, s0, Hq, Hkv, D = 10, 7, 2, 2, 1, 3
    ids = np.array([[1, 1, 1, 1, 2, 2, 2, 2, 2, 0]], np.int32)
    q, do = _rand((1, Hq, L, D), rng), _rand((1, Hq, L, D), rng)
    k, v = _rand((1, Hkv, S, D), rng), _rand((1, Hkv, S, D), rng)
    grads = orc.blockdiag_sdpa_backward(q, k, v, do, ids, s0, 0.7, True)

    def loss(qq, kk, vv):
        o, _ = orc.blockdiag_sdpa_forward(qq, kk, vv, ids, s0, 0.7, True)
        return float((o * do).sum())

    h = 1e-6
    for which, x in enumerate((q, k, v)):
        fd = np.zeros_like(x)
        for idx in np.ndindex(*x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            args_p = [q, k, v]
            args_m = [q, k, v]
            args_p[which], args_m[which] = xp, xm
            fd[idx] = (loss(*args_p) - loss(*args_m)) / (2 * h)
        np.testing.assert_allclose(grads[which], fd, rtol=1e-6, atol=1e-8)
