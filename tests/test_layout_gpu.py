"""GPU parity of the row-layout helpers against the layout oracle (bit-exact).

Covers: document ids from lengths (padding entries, zero-length documents,
empty rows, invalid lengths), document positions and validity, the position
check, and the key/value rows an interval of queries needs (with rows per
shard), at small sizes and at the 131072-token interval workload; row
lengths straddle the 4096-position chunks of the per-row scans.
"""
import numpy as np
import pytest
import torch

from oracle import layout as lay
from oracle import blockdiag as orc
from packed_sequence_block_gb300 import _native as N
from packed_sequence_block_gb300 import attention as A
from packed_sequence_block_gb300 import layout as LY
from packed_sequence_block_gb300.workloads import make_workload

pytestmark = pytest.mark.gpu


def _random_lens(rng, B, ndocs, S, pad_frac=0.3):
    lens = np.full((B, ndocs), -1000, np.int32)
    for b in range(B):
        budget = S
        for d in range(ndocs):
            if rng.random() < pad_frac:
                continue
            x = int(min(budget, rng.integers(0, max(1, S // max(1, ndocs // 2)) + 1)))
            lens[b, d] = x
            budget -= x
    return lens


@pytest.mark.parametrize("B,ndocs,S", [(1, 5, 256), (3, 7, 97), (2, 40, 4096), (2, 300, 4097),
                                       (1, 1, 1), (4, 0, 33), (1, 2000, 131072)])
def test_doc_ids_from_seq_lens_matches_oracle(cuda_lib, B, ndocs, S):
    rng = np.random.default_rng(B * 1000 + ndocs + S)
    lens = _random_lens(rng, B, ndocs, S)
    got = LY.doc_ids_from_seq_lens(torch.from_numpy(lens).cuda(), S).cpu().numpy()
    want = lay.doc_ids_from_seq_lens(lens, S) if ndocs else np.zeros((B, S), np.int32)
    np.testing.assert_array_equal(got, want)


def test_doc_ids_from_seq_lens_tiny_workload(cuda_lib):
    got = LY.doc_ids_from_seq_lens(torch.tensor([[37, 100, 1, 64, 54, -1000]]), 256).cpu()
    want = orc.doc_ids_from_cu_seqlens([0, 37, 137, 138, 202, 256], 256)
    np.testing.assert_array_equal(got.numpy()[0], want)


@pytest.mark.parametrize("lens,S", [([[3, -2, 1]], 8), ([[5, 4]], 8)])
def test_doc_ids_from_seq_lens_rejects(cuda_lib, lens, S):
    with pytest.raises(ValueError):
        LY.doc_ids_from_seq_lens(torch.tensor(lens, dtype=torch.int32), S)
    A.check_device_status()  # the error was consumed and reset


def _random_ids(rng, B, S):
    ids = np.zeros((B, S), np.int32)
    for b in range(B):
        p = 0
        while p < S:
            run = int(rng.integers(1, 40))
            ids[b, p:p + run] = rng.integers(0, 4)
            p += run
    return ids


@pytest.mark.parametrize("B,S", [(1, 1), (2, 37), (3, 4095), (2, 4096), (2, 4097), (1, 8193),
                                 (1, 131072)])
def test_position_ids_match_oracle(cuda_lib, B, S):
    rng = np.random.default_rng(B * 7 + S)
    ids = _random_ids(rng, B, S)
    pos, keep = LY.position_ids_from_doc_ids(torch.from_numpy(ids).cuda())
    wpos, wkeep = lay.position_ids_from_doc_ids(ids)
    np.testing.assert_array_equal(pos.cpu().numpy(), wpos)
    np.testing.assert_array_equal(keep.cpu().numpy(), wkeep)


@pytest.mark.parametrize("B,S", [(4, 64), (3, 4097), (2, 8193), (1, 131072)])
def test_validator_matches_oracle(cuda_lib, B, S):
    rng = np.random.default_rng(B * 11 + S)
    ids = _random_ids(rng, B, S)
    pos, keep = lay.position_ids_from_doc_ids(ids)
    pos = pos.astype(np.int32)
    # leave row 0 valid; break the others at a random column, sometimes twice
    for b in range(1, B):
        for _ in range(int(rng.integers(1, 3))):
            p = int(rng.integers(0, S))
            pos[b, p] = -3 if rng.random() < 0.3 else pos[b, p] + 2
    # row 0 becomes a shard that begins partway through a document, after left padding
    keep[0, :min(5, S)] = False
    got = LY.document_position_violations(torch.from_numpy(keep).cuda(),
                                          torch.from_numpy(pos).cuda()).cpu().numpy()
    np.testing.assert_array_equal(got, lay.validate_document_positions(keep, pos))


def test_validator_raises(cuda_lib):
    keep = torch.tensor([[True, True, False, True]], device="cuda")
    LY.validate_document_positions(keep, torch.tensor([[4, 5, 0, 0]], device="cuda"))
    with pytest.raises(ValueError, match="column 3"):
        LY.validate_document_positions(keep, torch.tensor([[4, 5, 0, 6]], device="cuda"))


def _check_range(ids_np, L, s0):
    ids = torch.from_numpy(ids_np).cuda()
    seg, sid, nseg = A.segment_cu_seqlens(ids)
    rng_, rows = LY.kv_needed_range(seg, sid, nseg, L, s0)
    rng_, rows = rng_.cpu().numpy(), rows.cpu().numpy()
    S = ids_np.shape[1]
    for b in range(ids_np.shape[0]):
        lo, hi = lay.kv_needed_range(ids_np[b], s0, L)
        assert (int(rng_[b, 0]), int(rng_[b, 1])) == (lo, hi), (b, s0, L)
        np.testing.assert_array_equal(rows[b], lay.kv_rows_per_shard(lo, hi, S, L))


@pytest.mark.parametrize("B,S,L", [(3, 64, 16), (2, 100, 30), (4, 4097, 1000), (1, 1, 1)])
def test_kv_needed_range_matches_oracle(cuda_lib, B, S, L):
    rng = np.random.default_rng(B + S + L)
    ids = _random_ids(rng, B, S)
    for s0 in sorted({0, S - L, int(rng.integers(0, S - L + 1))}):
        _check_range(ids, L, s0)


def test_kv_needed_range_interval_workload(cuda_lib):
    wl = make_workload("interval131k")
    ids = np.stack([orc.doc_ids_from_cu_seqlens(c, wl.S) for c in wl.cu])
    for s0 in wl.seq_starts:
        _check_range(ids, wl.L, s0)


def test_layout_entry_points_reject_bad_arguments(cuda_lib):
    seg, sid, nseg = A.segment_cu_seqlens(torch.zeros((1, 8), dtype=torch.int32, device="cuda"))
    r = torch.empty((1, 2), dtype=torch.int32, device="cuda")
    with pytest.raises(ValueError):
        N.bd_kv_needed_range(seg, sid, nseg, 1, 8, 4, 5, r)  # seq_start + L > S
    lens = torch.zeros((1, 8193), dtype=torch.int32, device="cuda")
    ids = torch.empty((1, 8), dtype=torch.int32, device="cuda")
    with pytest.raises(ValueError):
        N.bd_doc_ids_from_seq_lens(lens, 1, 8193, 8, -1000, ids)  # too many documents
