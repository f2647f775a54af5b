"""GPU plan (tile classifier + longest-first lists) against a brute-force mask.

The expected values come from the oracle's segments and the per-document causal
rule evaluated pair by pair; the plan buffer layout is the library's internal
one (int32 sections, 256-byte aligned, described in bd_internal.h).
"""
import numpy as np
import pytest
import torch

from oracle import blockdiag as orc
from packed_sequence_block_gb300 import attention as A

pytestmark = pytest.mark.gpu

PAD = 0x7FFFFFFF


def _layout(B, Hq, Hkv, L, S):
    a = lambda x: (x + 255) // 256 * 256  # noqa: E731
    G = Hq // Hkv
    QROWS = 128 if G % 2 == 0 else 256
    NQB, NKT = -(-L // QROWS), -(-S // 128)
    Lpad, Spad = NQB * QROWS, NKT * 128
    off = {}
    o = 0
    for name, n in (("qlo", B * Lpad), ("kend", B * Spad), ("fr", 2 * B * NQB),
                    ("br", 2 * B * NKT), ("fo", B * NQB), ("bo", B * NKT)):
        off[name] = (o, n)
        o = a(o + 4 * n)
    return off, QROWS, NQB, NKT, Lpad, Spad


def _mask(ids_row, seq_start, L):
    """allowed[i, j]: local query i (global seq_start+i) may attend key j."""
    S = ids_row.size
    seg, sid = orc.segment_cu_seqlens(ids_row)
    which = np.searchsorted(seg, np.arange(S), side="right") - 1
    t = seq_start + np.arange(L)
    j = np.arange(S)
    same = which[t][:, None] == which[None, :]
    return same & (j[None, :] <= t[:, None]) & (ids_row[t] != 0)[:, None]


CASES = [
    # rows of doc ids (built from cu lists), Hq, Hkv, L, seq_start
    ([[0, 37, 137, 138, 202, 256]], 256, 4, 2, 256, 0),
    ([[0, 300, 301, 700], [0, 1000]], 1000, 8, 8, 1000, 0),        # G = 1 (odd blocks)
    ([[0, 130, 900, 1500, 1900]], 2048, 6, 2, 700, 555),            # G = 3, interval
    ([[0, 64, 64, 400, 1024]], 1024, 4, 4, 256, 768),               # interval at the tail
    ([[0]], 512, 2, 1, 512, 0),                                     # all padding
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_plan_matches_brute_force(cuda_lib, case):
    cus, S, Hq, Hkv, L, s0 = CASES[case]
    B = len(cus)
    ids = np.stack([orc.doc_ids_from_cu_seqlens(c, S) for c in cus])
    tids = torch.from_numpy(ids).cuda()
    seg, sid, nseg = A.segment_cu_seqlens(tids)
    plan = A.make_plan(seg, sid, nseg, Hq, Hkv, L, s0)
    A.check_device_status()
    raw = plan.cpu().numpy().view(np.int32)
    off, QROWS, NQB, NKT, Lpad, Spad = _layout(B, Hq, Hkv, L, S)
    sec = {k: raw[o // 4:o // 4 + n] for k, (o, n) in off.items()}
    qlo = sec["qlo"].reshape(B, Lpad)
    kend = sec["kend"].reshape(B, Spad)
    fr = sec["fr"].reshape(B * NQB, 2)
    br = sec["br"].reshape(B * NKT, 2)
    for b in range(B):
        sg, si = orc.segment_cu_seqlens(ids[b])
        which = np.searchsorted(sg, np.arange(S), side="right") - 1
        for i in range(Lpad):
            t = s0 + i
            exp = PAD if (i >= L or si[which[t]] == 0) else sg[which[t]]
            assert qlo[b, i] == exp, (b, i)
        for p in range(Spad):
            exp = p if (p >= S or si[which[p]] == 0) else sg[which[p] + 1]
            assert kend[b, p] == exp, (b, p)
        m = _mask(ids[b], s0, L)
        mp = np.zeros((Lpad, Spad), bool)
        mp[:L, :S] = m
        for qb in range(NQB):
            rows = mp[qb * QROWS:(qb + 1) * QROWS]
            tiles = [kt for kt in range(NKT) if rows[:, kt * 128:(kt + 1) * 128].any()]
            lo, hi = fr[b * NQB + qb]
            if tiles:
                assert (lo, hi) == (min(tiles), max(tiles))
            else:
                assert hi < lo
        for kt in range(NKT):
            cols = mp[:, kt * 128:(kt + 1) * 128]
            qts = [qt for qt in range(-(-L // 128)) if cols[qt * 128:(qt + 1) * 128].any()]
            lo, hi = br[b * NKT + kt]
            if qts:
                assert (lo, hi) == (min(qts), max(qts))
            else:
                assert hi < lo
    for order, rng_ in ((sec["fo"], fr), (sec["bo"], br)):
        assert sorted(order.tolist()) == list(range(order.size))
        cost = np.maximum(0, rng_[order, 1] - rng_[order, 0] + 1)
        assert np.all(np.diff(cost) <= 0), "work list is not longest-first"
