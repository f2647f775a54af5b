"""GPU plan (tile classifier + ordered work lists) against a brute-force mask.

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
    # the per-tile range searches at their edges: boundaries on tile edges,
    # empty documents on a tile edge with the interval starting mid-document
    # and padding after it, an interval wholly in padding, one-token documents
    ([[0, 128, 256, 384, 512]], 512, 2, 2, 512, 0),
    ([[0, 128, 128, 128, 300, 1000]], 1024, 4, 2, 600, 200),
    ([[0, 100]], 1024, 2, 1, 500, 300),
    ([[0, 1, 2, 3, 640], [0, 639, 640]], 640, 3, 3, 640, 0),
    # a long document: the forward list goes longest first
    ([[0, 1900, 2048]], 2048, 2, 2, 2048, 0),
    # at the order rule's threshold: a query block reaching 8 key tiles keeps
    # position order, one reaching 9 goes longest first
    ([[0, 1024, 1100]], 1100, 2, 2, 1100, 0),
    ([[0, 1025, 1100]], 1100, 2, 2, 1100, 0),
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
    fo, bo = sec["fo"], sec["bo"]
    assert fo.tolist() == _forward_order(fr), "forward work list order"
    assert bo.tolist() == _document_order(br, NKT), "backward work list is not by document"


# Longest forward unit (key tiles) that still keeps the list in position order.
SHORT_FWD_UNIT = 8


def _forward_order(fr):
    """Forward order: longest first, ties by index; position order when no
    query block reaches more than SHORT_FWD_UNIT key tiles."""
    cost = np.maximum(0, fr[:, 1] - fr[:, 0] + 1)
    if cost.max(initial=0) <= SHORT_FWD_UNIT:
        return list(range(len(fr)))
    return sorted(range(len(fr)), key=lambda i: (-int(cost[i]), i))


def _document_order(br, NKT):
    """Backward order: each document's key tiles together (a run of tiles of one
    row reaching the same last query tile), longest first within it; documents
    by the cost of their first tile, largest first; empty tiles last; ties by
    index."""
    keys, head = [], -1
    for i, (lo, hi) in enumerate(br.tolist()):
        plo, phi = br[i - 1].tolist() if i else (0, -1)
        if hi < lo or i % NKT == 0 or phi < plo or phi != hi:
            head = i
        size = 0 if hi < lo else int(br[head, 1] - br[head, 0] + 1)
        keys.append((-size, i))
    return [i for _, i in sorted(keys)]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_single_call_plan_equals_planned(cuda_lib, case):
    """The single-call forward builds its plan from the boundaries inside its
    workspace (after a 256-byte record); every section but the work counters
    must equal the plan built from segments."""
    cus, S, Hq, Hkv, L, s0 = CASES[case]
    B = len(cus)
    ids = np.stack([orc.doc_ids_from_cu_seqlens(c, S) for c in cus])
    seg, sid, nseg = A.segment_cu_seqlens(torch.from_numpy(ids).cuda())
    plan = A.make_plan(seg, sid, nseg, Hq, Hkv, L, s0)
    g = torch.Generator().manual_seed(case)
    D = 64
    q = torch.randn((B, Hq, L, D), generator=g).to(torch.bfloat16).cuda()
    k = torch.randn((B, Hkv, S, D), generator=g).to(torch.bfloat16).cuda()
    v = torch.randn((B, Hkv, S, D), generator=g).to(torch.bfloat16).cuda()
    cu, rp = A.cu_csr(cus, "cuda")
    _, _, ws = A.attn_forward_cu(q, k, v, cu, rp, s0, None, Hq != Hkv)
    A.check_device_status()
    off, *_ = _layout(B, Hq, Hkv, L, S)
    planned = plan.cpu().numpy().view(np.int32)
    single = ws.cpu().numpy()[256:256 + plan.numel()].view(np.int32)
    for name, (o, n) in off.items():
        assert np.array_equal(single[o // 4:o // 4 + n], planned[o // 4:o // 4 + n]), name
