"""GPU parity of the index kernels: document ids and segments, bit-exact against the oracle."""
import numpy as np
import pytest
import torch

from oracle import blockdiag as orc
from packed_sequence_block_gb300 import attention as A
from packed_sequence_block_gb300 import _native as N
from packed_sequence_block_gb300.workloads import WORKLOADS, make_workload, random_cu

pytestmark = pytest.mark.gpu


def _check_rows(cu_rows, S):
    ids = A.doc_ids_from_cu_seqlens([np.asarray(c, np.int32) for c in cu_rows], S)
    A.check_device_status()
    got = ids.cpu().numpy()
    seg, sid, nseg = A.segment_cu_seqlens(ids)
    seg, sid, nseg = seg.cpu().numpy(), sid.cpu().numpy(), nseg.cpu().numpy()
    for b, cu in enumerate(cu_rows):
        exp = orc.doc_ids_from_cu_seqlens(cu, S)
        np.testing.assert_array_equal(got[b], exp)
        es, ei = orc.segment_cu_seqlens(exp)
        n = int(nseg[b])
        assert n == ei.size
        np.testing.assert_array_equal(seg[b, :n + 1], es)
        np.testing.assert_array_equal(sid[b, :n], ei)


@pytest.mark.parametrize("name", WORKLOADS)
def test_workload_ids_and_segments(cuda_lib, name):
    wl = make_workload(name, 0)
    _check_rows(wl.cu, wl.S)


@pytest.mark.parametrize("seed", range(24))
def test_random_boundaries(cuda_lib, seed):
    rng = np.random.default_rng(1000 + seed)
    S = int(rng.choice([1, 2, 7, 128, 129, 1000, 4095, 4096, 4097, 9001]))
    B = int(rng.integers(1, 4))
    rows = [random_cu(rng, S, max_docs=int(rng.integers(1, 40))) for _ in range(B)]
    _check_rows(rows, S)


def test_all_padding_and_empty_documents(cuda_lib):
    _check_rows([[0], [0, 0, 0], [0, 5, 5, 5, 9]], 16)


def test_invalid_boundaries_report_status(cuda_lib):
    S = 32
    rows = [np.array([0, 8, 4, 16], np.int32), np.array([0, 40], np.int32),
            np.array([3, 9], np.int32), np.array([0, 10, 32], np.int32)]
    ids = A.doc_ids_from_cu_seqlens(rows, S)
    code = N.bd_get_device_status(A.device_status_word())
    A.device_status_word().zero_()
    assert code == N.BD_ERR_INVALID_ARG
    got = ids.cpu().numpy()
    assert np.all(got[:3] == 0)
    np.testing.assert_array_equal(got[3], orc.doc_ids_from_cu_seqlens(rows[3], S))


@pytest.mark.parametrize("seed", range(8))
def test_segments_of_arbitrary_ids(cuda_lib, seed):
    rng = np.random.default_rng(seed)
    S = int(rng.integers(1, 20000))
    runs = rng.integers(1, 300, size=S)
    vals = rng.integers(0, 4, size=S)  # repeats of earlier ids and interior padding
    ids = np.repeat(vals, runs)[:S].astype(np.int32)
    t = torch.from_numpy(ids).cuda()[None]
    seg, sid, nseg = A.segment_cu_seqlens(t)
    es, ei = orc.segment_cu_seqlens(ids)
    n = int(nseg.item())
    assert n == ei.size
    np.testing.assert_array_equal(seg[0, :n + 1].cpu().numpy(), es)
    np.testing.assert_array_equal(sid[0, :n].cpu().numpy(), ei)
