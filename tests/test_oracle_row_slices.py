"""Pins for the oracle's row slicing.

The oracle computes one segment at a time and, to bound memory, cuts a
segment's query rows into slices once rows x keys would exceed a budget
(``oracle.blockdiag._ROW_BUDGET``).  At the default budget no workload small
enough for the pins reaches that branch, so here the budget is shrunk until
every segment is cut into many slices (down to one row each), and the sliced
results must equal

* the unsliced results of the same oracle (to 1e-12), and
* an independent dense statement: the mask of cp_blockdiag_sdpa (page
  "nemo_automodel.components.distributed.blockdiag_cp": the query at global
  position t attends keys j <= t of its own segment, padding attends
  nothing) written out element by element in pure Python, then masked
  softmax attention and its gradients by torch autograd in fp64.

The cases cover several documents in a row, interior padding, a query
interval that starts inside a document, GQA, two rows, and dropout (the
mask's query and key positions in a later slice).
"""
import math

import numpy as np
import pytest
import torch

from oracle import blockdiag as orc
from oracle import dropout as dro

CASES = {
    # name: (ids rows, seq_start, L, Hq, Hkv, D, dropout (p, seed, offset) or None)
    "three_docs_interior_pad": (
        [[1] * 23 + [2] * 17 + [0] * 3 + [3] * 9], 0, 52, 2, 2, 4, None),
    "interval_mid_document_gqa": (
        [[1] * 7 + [2] * 30 + [0] * 2 + [3] * 13], 10, 30, 4, 2, 3, None),
    "two_rows_gqa": (
        [[5] * 26 + [0] * 4 + [6] * 10, [1] * 40], 3, 33, 3, 1, 2, None),
    "dropout_interval": (
        [[1] * 19 + [2] * 21 + [0] * 2], 6, 34, 2, 1, 3, (0.3, 0x1234_5678_9ABC, 7)),
}
BUDGETS = [5, 37, 256]


def _dense_mask(ids, seq_start, L):
    """[B, L, S] booleans from the rule, one element at a time."""
    B, S = len(ids), len(ids[0])
    m = np.zeros((B, L, S), bool)
    for b in range(B):
        for i in range(L):
            t = seq_start + i
            if ids[b][t] == 0:
                continue
            for j in range(t + 1):
                m[b, i, j] = all(ids[b][x] == ids[b][t] for x in range(j, t + 1))
    return m


def _dense_reference(q, k, v, do, ids, seq_start, G, drop):
    """out, lse, dq, dk, dv by a dense masked softmax and torch autograd (fp64)."""
    B, Hq, L, D = q.shape
    S = k.shape[2]
    scale = D ** -0.5
    mask = torch.from_numpy(_dense_mask(ids, seq_start, L))[:, None]  # [B, 1, L, S]
    live = mask.any(-1, keepdim=True)                                   # rows with keys
    tq, tk, tv = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (q, k, v))
    kk = tk.repeat_interleave(G, dim=1)
    vv = tv.repeat_interleave(G, dim=1)
    s = scale * tq @ kk.transpose(-1, -2)
    s = s.masked_fill(~(mask | ~live), -math.inf)  # rows without keys stay finite, zeroed below
    p = torch.softmax(s, dim=-1) * live
    lse = torch.where(live[..., 0], torch.logsumexp(s, dim=-1), -math.inf)
    if drop is not None:
        pdrop, seed, offset = drop
        keep = np.zeros((B, Hq, L, S))
        for b in range(B):
            for h in range(Hq):
                keep[b, h] = dro.keep_mask(b * Hq + h, np.arange(L) + seq_start, np.arange(S),
                                           seed, offset, pdrop)
        p = p * torch.from_numpy(keep) * dro.keep_scale(pdrop)
    out = p @ vv
    out.backward(torch.tensor(do, dtype=torch.float64))
    f = lambda t: t.detach().numpy()  # noqa: E731
    return f(out), f(lse), f(tq.grad), f(tk.grad), f(tv.grad)


def _inputs(case, seed=3):
    rows, seq_start, L, Hq, Hkv, D, drop = case
    rng = np.random.default_rng(seed)
    B, S = len(rows), len(rows[0])
    q, do = rng.standard_normal((B, Hq, L, D)), rng.standard_normal((B, Hq, L, D))
    k, v = rng.standard_normal((B, Hkv, S, D)), rng.standard_normal((B, Hkv, S, D))
    return np.asarray(rows, np.int32), q, k, v, do


def _run(mod, ids, q, k, v, do, seq_start, gqa, drop):
    kw = {}
    if drop is not None:
        kw = dict(dropout_p=drop[0], seed=drop[1], offset=drop[2])
    out, lse = mod.blockdiag_sdpa_forward(q, k, v, ids, seq_start, None, gqa, **kw)
    dq, dk, dv = mod.blockdiag_sdpa_backward(q, k, v, do, ids, seq_start, None, gqa,
                                             out=out, lse=lse, **kw)
    return out, lse, dq, dk, dv


def _close(name, got, exp, tol=1e-12):
    got, exp = np.asarray(got), np.asarray(exp)
    assert np.array_equal(np.isneginf(got), np.isneginf(exp)), f"{name}: -inf pattern"
    fin = np.isfinite(exp)
    np.testing.assert_allclose(got[fin], exp[fin], rtol=tol, atol=tol, err_msg=name)


def check_sliced_oracle(mod, name, budget):
    """Sliced results of oracle module ``mod`` against its unsliced results and the
    dense statement; raises AssertionError on a mismatch."""
    rows, seq_start, L, Hq, Hkv, D, drop = CASES[name]
    ids, q, k, v, do = _inputs(CASES[name])
    gqa = Hq != Hkv
    whole = _run(mod, ids, q, k, v, do, seq_start, gqa, drop)
    saved = mod._ROW_BUDGET
    mod._ROW_BUDGET = budget
    try:
        sliced = _run(mod, ids, q, k, v, do, seq_start, gqa, drop)
    finally:
        mod._ROW_BUDGET = saved
    dense = _dense_reference(q, k, v, do, rows, seq_start, Hq // Hkv, drop)
    for label, a, w, d in zip(("out", "lse", "dq", "dk", "dv"), sliced, whole, dense):
        _close(f"{name} budget {budget} {label} vs unsliced", a, w)
        _close(f"{name} budget {budget} {label} vs dense", a, d, tol=1e-10)


def test_small_budgets_really_slice(monkeypatch):
    """The budgets below cut every case's segments into several slices."""
    monkeypatch.setattr(orc, "_ROW_BUDGET", 37)
    assert list(orc._row_slices(10, 37, 37)) == [(t, t + 1) for t in range(10, 37)]
    monkeypatch.setattr(orc, "_ROW_BUDGET", 256)
    assert list(orc._row_slices(0, 40, 40)) == [(0, 6), (6, 12), (12, 18), (18, 24),
                                                (24, 30), (30, 36), (36, 40)]


@pytest.mark.parametrize("budget", BUDGETS)
@pytest.mark.parametrize("name", sorted(CASES))
def test_sliced_oracle_matches_unsliced_and_dense(name, budget):
    check_sliced_oracle(orc, name, budget)
