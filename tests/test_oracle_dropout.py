"""Pins for attention dropout in the oracle.

Page "nemo_automodel.components.distributed.blockdiag_cp", cp_blockdiag_sdpa
(dropout_p).  The generator (Philox4x32-10, Salmon et al., SC'11) is pinned here by
properties (bijectivity, uniform words, the drop rate, independent
neighbouring keys) and, on a GPU, word for word against cuRAND's
implementation (test_oracle_philox_gpu.py); the dropout
arithmetic by exact reductions: p = 0, a dense element-by-element restatement
with the mask written out, the expectation over masks, finite differences
with the mask fixed, and interval invariance.
"""
import math

import numpy as np
import pytest

from oracle import blockdiag as orc
from oracle import dropout as dro


# ---------------------------------------------------------------- generator

def test_philox_is_a_bijection_on_counters():
    c = np.arange(1 << 16, dtype=np.int64)
    w = dro.philox4x32_10(c & 0xFF, c >> 8, 7, 0, 0x0123456789ABCDEF)
    packed = {tuple(int(x[i]) for x in w) for i in range(c.size)}
    assert len(packed) == c.size


def test_philox_words_are_uniform():
    c = np.arange(1 << 15, dtype=np.int64)
    words = np.concatenate([x.astype(np.float64) for x in dro.philox4x32_10(c, 3, 5, 11, 42)])
    u = words / 2.0 ** 32
    n = u.size
    assert abs(u.mean() - 0.5) < 4 * math.sqrt(1 / 12 / n)
    counts = np.histogram(u, bins=16, range=(0.0, 1.0))[0]
    chi2 = float(((counts - n / 16) ** 2 / (n / 16)).sum())
    assert chi2 < 45.0  # 15 degrees of freedom: p ~ 1e-4


def test_philox_depends_on_every_input():
    base = dro.philox4x32_10(1, 2, 3, 4, 5)
    for args in ((0, 2, 3, 4, 5), (1, 0, 3, 4, 5), (1, 2, 0, 4, 5), (1, 2, 3, 0, 5),
                 (1, 2, 3, 4, 6), (1, 2, 3, 4, 5 + (1 << 32))):
        assert tuple(dro.philox4x32_10(*args)) != tuple(base)


@pytest.mark.parametrize("p", [0.1, 0.5, 0.9])
def test_drop_rate(p):
    keep = dro.keep_mask(3, np.arange(200), np.arange(1000), 99, 0, p)
    n = keep.size
    rate = 1.0 - keep.mean()
    assert abs(rate - p) < 5 * math.sqrt(p * (1 - p) / n)


def test_threshold_and_p_zero():
    assert dro.drop_threshold(0.0) == 0
    assert dro.drop_threshold(0.5) == 1 << 15
    assert dro.drop_threshold(0.3) == 19660  # 0.3 * 65536 = 19660.8
    assert dro.drop_threshold(2.0 ** -17) == 0  # below the 16-bit grain: nothing drops
    assert dro.keep_scale(0.25) == 4.0 / 3.0
    assert dro.keep_scale(0.3) == 1.0 / (1.0 - 19660 / 65536)
    assert dro.keep_mask(0, np.arange(5), np.arange(9), 1, 0, 0.0).all()
    assert dro.keep_mask(0, np.arange(5), np.arange(9), 1, 0, 2.0 ** -17).all()
    with pytest.raises(ValueError):
        dro.drop_threshold(1.0)


def test_neighbouring_keys_are_independent():
    """Each key of an 8-key block draws its own 16 bits: two keys sharing a
    value (or a word's half used twice) would correlate their decisions."""
    p = 0.5
    keep = dro.keep_mask(2, np.arange(256), np.arange(512), 7, 1, p)
    for d in range(1, 9):
        both = (keep[:, :-d] & keep[:, d:]).mean()
        n = keep[:, d:].size
        assert abs(both - 0.25) < 5 * math.sqrt(0.25 * 0.75 / n), d
    # the same key across neighbouring queries too
    both = (keep[:-1] & keep[1:]).mean()
    assert abs(both - 0.25) < 5 * math.sqrt(0.25 * 0.75 / keep[1:].size)


# ---------------------------------------------------------------- attention with dropout

def _rand(shape, rng):
    return rng.standard_normal(shape)


def _dense_dropout_forward(q, k, v, ids, s0, scale, G, p, seed, offset):
    """Element by element: weights from the definition, then the mask written out."""
    B, Hq, L, D = q.shape
    S = k.shape[2]
    out = np.zeros((B, Hq, L, D))
    for b in range(B):
        for h in range(Hq):
            g = h // G
            for i in range(L):
                t = s0 + i
                if ids[b][t] == 0:
                    continue
                allowed = [j for j in range(S)
                           if j <= t and all(ids[b][x] == ids[b][t] for x in range(j, t + 1))]
                s = {j: scale * float(q[b, h, i] @ k[b, g, j]) for j in allowed}
                z = sum(math.exp(x) for x in s.values())
                for j in allowed:
                    keep = dro.keep_mask(b * Hq + h, [t], [j], seed, offset, p)[0, 0]
                    p_eff = math.floor(p * 65536) / 65536  # p on the 16-bit grain
                    w = math.exp(s[j]) / z * (1.0 / (1.0 - p_eff) if keep else 0.0)
                    out[b, h, i] += w * v[b, g, j]
    return out


CASES = [
    ([[1, 1, 1, 2, 2, 3, 3, 3, 3, 0, 0]], 0, 11, 2, 1, 3),
    ([[4, 4, 4, 4, 4, 7, 7, 7, 0, 0, 9, 9]], 3, 6, 4, 2, 2),
]


@pytest.mark.parametrize("case", CASES)
def test_dropout_forward_matches_dense_statement(case):
    rows, s0, L, Hq, Hkv, D = case
    rng = np.random.default_rng(31)
    ids = np.asarray(rows, np.int32)
    B, S = ids.shape
    q, k, v = _rand((B, Hq, L, D), rng), _rand((B, Hkv, S, D), rng), _rand((B, Hkv, S, D), rng)
    out, lse = orc.blockdiag_sdpa_forward(q, k, v, ids, s0, None, Hq != Hkv, 0.3, 1234, 5)
    want = _dense_dropout_forward(q, k, v, ids, s0, D ** -0.5, Hq // Hkv, 0.3, 1234, 5)
    np.testing.assert_allclose(out, want, rtol=1e-12, atol=1e-12)
    # the log-sum-exp is the softmax's, untouched by dropout
    _, lse0 = orc.blockdiag_sdpa_forward(q, k, v, ids, s0, None, Hq != Hkv)
    np.testing.assert_array_equal(lse, lse0)


def test_dropout_zero_is_no_dropout():
    rows, s0, L, Hq, Hkv, D = CASES[0]
    rng = np.random.default_rng(32)
    ids = np.asarray(rows, np.int32)
    B, S = ids.shape
    q, k, v = _rand((B, Hq, L, D), rng), _rand((B, Hkv, S, D), rng), _rand((B, Hkv, S, D), rng)
    a = orc.blockdiag_sdpa_forward(q, k, v, ids, s0, None, True, 0.0, 77, 3)
    b = orc.blockdiag_sdpa_forward(q, k, v, ids, s0, None, True)
    np.testing.assert_array_equal(a[0], b[0])


def test_dropout_is_unbiased_over_masks():
    rows, s0, L, Hq, Hkv, D = CASES[0]
    rng = np.random.default_rng(33)
    ids = np.asarray(rows, np.int32)
    B, S = ids.shape
    q, k, v = _rand((B, Hq, L, D), rng), _rand((B, Hkv, S, D), rng), _rand((B, Hkv, S, D), rng)
    ref, _ = orc.blockdiag_sdpa_forward(q, k, v, ids, s0, None, True)
    n = 3000
    acc = np.zeros_like(ref)
    sq = np.zeros_like(ref)
    for seed in range(n):
        o, _ = orc.blockdiag_sdpa_forward(q, k, v, ids, s0, None, True, 0.25, seed, 0)
        acc += o
        sq += o * o
    mean = acc / n
    sd = np.sqrt(np.maximum(sq / n - mean * mean, 0.0) / n) + 1e-12
    assert np.all(np.abs(mean - ref) <= 5 * sd + 1e-9)


def test_dropout_backward_matches_finite_differences():
    rng = np.random.default_rng(34)
    S, L, s0, Hq, Hkv, D = 10, 7, 2, 2, 1, 3
    ids = np.array([[1, 1, 1, 1, 2, 2, 2, 2, 2, 0]], np.int32)
    q, do = _rand((1, Hq, L, D), rng), _rand((1, Hq, L, D), rng)
    k, v = _rand((1, Hkv, S, D), rng), _rand((1, Hkv, S, D), rng)
    p, seed, off = 0.35, 2024, 9
    grads = orc.blockdiag_sdpa_backward(q, k, v, do, ids, s0, 0.7, True, dropout_p=p, seed=seed,
                                        offset=off)

    def loss(qq, kk, vv):
        o, _ = orc.blockdiag_sdpa_forward(qq, kk, vv, ids, s0, 0.7, True, p, seed, off)
        return float((o * do).sum())

    h = 1e-6
    for which, x in enumerate((q, k, v)):
        fd = np.zeros_like(x)
        for idx in np.ndindex(*x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            args_p, args_m = [q, k, v], [q, k, v]
            args_p[which], args_m[which] = xp, xm
            fd[idx] = (loss(*args_p) - loss(*args_m)) / (2 * h)
        np.testing.assert_allclose(grads[which], fd, rtol=1e-6, atol=1e-8)


def test_dropout_intervals_concatenate_to_full_rows():
    rng = np.random.default_rng(35)
    S, Hq, Hkv, D = 12, 2, 1, 3
    ids = np.array([[1, 1, 1, 1, 1, 2, 2, 2, 2, 2, 2, 0]], np.int32)
    q, k, v = _rand((1, Hq, S, D), rng), _rand((1, Hkv, S, D), rng), _rand((1, Hkv, S, D), rng)
    full, _ = orc.blockdiag_sdpa_forward(q, k, v, ids, 0, None, True, 0.4, 5, 1)
    parts = [orc.blockdiag_sdpa_forward(q[:, :, s:s + 4], k, v, ids, s, None, True, 0.4, 5, 1)[0]
             for s in (0, 4, 8)]
    np.testing.assert_allclose(np.concatenate(parts, axis=2), full, rtol=0, atol=1e-14)


def test_dropout_slice_draws_the_whole_problems_mask():
    """A document and a subset of heads, cut out with their planes and positions,
    give the whole problem's values (the slice form the sampled checks use)."""
    rng = np.random.default_rng(36)
    B, Hq, Hkv, S, D = 2, 4, 2, 14, 3
    ids = np.array([[1] * 5 + [2] * 6 + [0] * 3, [3] * 9 + [4] * 5], np.int32)
    q, do = _rand((B, Hq, S, D), rng), _rand((B, Hq, S, D), rng)
    k, v = _rand((B, Hkv, S, D), rng), _rand((B, Hkv, S, D), rng)
    p, seed, off = 0.4, (7 << 40) | 3, 2
    out, lse = orc.blockdiag_sdpa_forward(q, k, v, ids, 0, None, True, p, seed, off)
    dq, dk, dv = orc.blockdiag_sdpa_backward(q, k, v, do, ids, 0, None, True, out=out, lse=lse,
                                             dropout_p=p, seed=seed, offset=off)
    b, a, e, heads = 0, 5, 11, [2, 3]  # document 2 of row 0, kv head 1
    r0 = 7
    sl = (slice(b, b + 1), heads)
    planes = [[b * Hq + h for h in heads]]
    ones = np.ones((1, e - a), np.int32)
    so, sls = orc.blockdiag_sdpa_forward(q[sl][:, :, r0:e], k[b:b + 1, 1:2, a:e],
                                         v[b:b + 1, 1:2, a:e], ones, r0 - a, None, True, p, seed,
                                         off, mask_planes=planes, mask_pos0=a)
    np.testing.assert_allclose(so, out[sl][:, :, r0:e], rtol=0, atol=1e-13)
    np.testing.assert_allclose(sls, lse[sl][:, :, r0:e], rtol=0, atol=1e-13)
    # dk/dv of the document's keys from all of its queries
    _, sdk, sdv = orc.blockdiag_sdpa_backward(q[sl][:, :, a:e], k[b:b + 1, 1:2, a:e],
                                              v[b:b + 1, 1:2, a:e], do[sl][:, :, a:e], ones, 0,
                                              None, True, dropout_p=p, seed=seed, offset=off,
                                              mask_planes=planes, mask_pos0=a)
    np.testing.assert_allclose(sdk[0, 0], dk[b, 1, a:e], rtol=0, atol=1e-12)
    np.testing.assert_allclose(sdv[0, 0], dv[b, 1, a:e], rtol=0, atol=1e-12)
    # and a wrong plane draws another mask
    wrong, _ = orc.blockdiag_sdpa_forward(q[sl][:, :, r0:e], k[b:b + 1, 1:2, a:e],
                                          v[b:b + 1, 1:2, a:e], ones, r0 - a, None, True, p,
                                          seed, off, mask_planes=[[0, 1]], mask_pos0=a)
    assert np.abs(wrong - out[sl][:, :, r0:e]).max() > 1e-3
