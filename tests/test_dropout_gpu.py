"""GPU parity of attention dropout against the oracle.

Page "nemo_automodel.components.distributed.blockdiag_cp", cp_blockdiag_sdpa
(dropout_p).  The keep mask is an integer decision, so it is compared bit for
bit: with V (forward) or dO (backward) set to one-hot rows over the
positions of a document, each output element is nonzero exactly when one
weight was kept, which reads the kernels' mask back element by element.  The
values are compared with the fp64 oracle under the same mask at the parity
bar (small cases in full, the 8192-token workload on sampled rows).
"""
import zlib

import numpy as np
import pytest
import torch

from _gpu_common import (assert_close, assert_lse, gpu_forward_backward, rand_bf16,
                         sampled_checks, to64)
from oracle import blockdiag as orc
from oracle import dropout as dro
from packed_sequence_block_gb300 import attention as A
from packed_sequence_block_gb300.workloads import make_qkv_do, make_workload

pytestmark = pytest.mark.gpu

SEED = 0x9E3779B97F4A7C15  # both 32-bit key words non-zero


def _ids(cu_rows, S):
    return np.stack([orc.doc_ids_from_cu_seqlens(c, S) for c in cu_rows])


def _aligned_docs(B, S, W, pad_tail):
    """Documents of exactly W tokens starting at multiples of W; the last
    ``pad_tail`` tokens of row 1 are padding."""
    ids = np.zeros((B, S), np.int32)
    for b in range(B):
        for d in range(S // W):
            ids[b, d * W:(d + 1) * W] = d + 1
    if B > 1 and pad_tail:
        ids[1, S - pad_tail:] = 0
    return ids


def _one_hot_rows(B, H, n, W, pos0=0):
    """bf16 [B, H, n, W]: row r is the unit vector of column (pos0 + r) mod W."""
    x = torch.zeros((B, H, n, W), dtype=torch.bfloat16)
    cols = (torch.arange(n) + pos0) % W
    x[:, :, torch.arange(n), cols] = 1.0
    return x.cuda()


@pytest.mark.parametrize("D,s0,L,p", [(64, 0, 1024, 0.3), (128, 0, 1024, 0.5),
                                      (64, 192, 450, 0.2), (128, 256, 640, 0.75)])
def test_forward_mask_bit_exact(cuda_lib, D, s0, L, p):
    B, Hq, Hkv, S, W = 2, 4, 2, 1024, D
    ids = _aligned_docs(B, S, W, pad_tail=100)
    g = torch.Generator().manual_seed(D + s0)
    q, k = rand_bf16((B, Hq, L, D), g), rand_bf16((B, Hkv, S, D), g)
    v = _one_hot_rows(B, Hkv, S, W)
    do = rand_bf16((B, Hq, L, D), g)
    out, lse, *_ = gpu_forward_backward(q, k, v, do, torch.from_numpy(ids).cuda(), s0,
                                        dropout=(p, SEED, 11))
    got = (out.float().cpu().numpy() != 0.0)
    t = np.arange(s0, s0 + L)
    cols = np.arange(W)
    for b in range(B):
        for h in range(Hq):
            keep = dro.keep_mask(b * Hq + h, t, np.arange(S), SEED, 11, p)  # [L, S]
            j = (t // W * W)[:, None] + cols[None, :]                      # key of each column
            allowed = (j <= t[:, None]) & (ids[b][t] != 0)[:, None]
            want = allowed & np.take_along_axis(keep, j, axis=1)
            np.testing.assert_array_equal(got[b, h], want, err_msg=f"b={b} h={h}")
    # padding rows: zero output, -inf lse
    assert np.all(np.isneginf(lse[1, :, max(0, S - 100 - s0):].cpu().numpy()))


@pytest.mark.parametrize("D,s0,L,p", [(64, 0, 1024, 0.3), (128, 0, 1024, 0.6),
                                      (64, 320, 500, 0.45)])
def test_backward_mask_bit_exact(cuda_lib, D, s0, L, p):
    """dv = rp (P o M)^T dO with one-hot dO rows: dv[j, c] != 0 iff query
    (start of j's document) + c attends j and its weight was kept."""
    B, H, S, W = 2, 3, 1024, D
    ids = _aligned_docs(B, S, W, pad_tail=0)
    g = torch.Generator().manual_seed(7 * D + s0)
    q, k, v = rand_bf16((B, H, L, D), g), rand_bf16((B, H, S, D), g), rand_bf16((B, H, S, D), g)
    do = _one_hot_rows(B, H, L, W, pos0=s0)
    _, _, _, _, dv = gpu_forward_backward(q, k, v, do, torch.from_numpy(ids).cuda(), s0,
                                          dropout=(p, SEED, 3))
    got = (dv.float().cpu().numpy() != 0.0)
    j = np.arange(S)
    cols = np.arange(W)
    tq = (j // W * W)[:, None] + cols[None, :]       # the query feeding column c of key j
    in_interval = (tq >= s0) & (tq < s0 + L)
    for b in range(B):
        for h in range(H):
            keep = dro.keep_mask(b * H + h, np.arange(S), j, SEED, 3, p)  # [t, j]
            kept = keep[tq, j[:, None]]
            want = (tq >= j[:, None]) & in_interval & kept
            np.testing.assert_array_equal(got[b, h], want, err_msg=f"b={b} h={h}")


def _compare(ids, q, k, v, do, s0, drop, tag):
    gqa = q.shape[1] != k.shape[1]
    out, lse, dq, dk, dv = gpu_forward_backward(q, k, v, do, torch.from_numpy(ids).cuda(), s0,
                                                None, gqa, dropout=drop)
    p, seed, off = drop
    eo, el = orc.blockdiag_sdpa_forward(q, k, v, ids, s0, None, gqa, p, seed, off)
    edq, edk, edv = orc.blockdiag_sdpa_backward(q, k, v, do, ids, s0, None, gqa, out=eo, lse=el,
                                                dropout_p=p, seed=seed, offset=off)
    assert_close(f"{tag} out", to64(out), eo)
    assert_lse(f"{tag} lse", to64(lse), el)
    assert_close(f"{tag} dq", to64(dq), edq)
    assert_close(f"{tag} dk", to64(dk), edk)
    assert_close(f"{tag} dv", to64(dv), edv)


CASES = {
    # name: (cu rows, S, L, seq_start, Hq, Hkv, D, p)
    "tiny_p0.1": ([[0, 37, 137, 138, 202, 256]], 256, 256, 0, 4, 2, 64, 0.1),
    "g3_ragged_d128_p0.5": ([[0, 17, 260, 517], [0, 400]], 517, 517, 0, 6, 2, 128, 0.5),
    "g8_d64_onedoc_p0.2": ([[0, 1500]], 1500, 1500, 0, 8, 1, 64, 0.2),
    "interval_unaligned_p0.3": ([[0, 150, 600, 1024]], 1024, 300, 200, 4, 1, 64, 0.3),
    "interval_aligned_p0.9": ([[0, 700, 1300, 2048]], 2048, 256, 768, 4, 2, 128, 0.9),
    "all_pad_row_p0.25": ([[0, 90, 256], [0]], 256, 256, 0, 2, 1, 128, 0.25),
    "one_token_docs_p0.5": ([list(range(0, 257))], 256, 256, 0, 2, 2, 64, 0.5),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_dropout_small_cases(cuda_lib, name):
    cu_rows, S, L, s0, Hq, Hkv, D, p = CASES[name]
    B = len(cu_rows)
    g = torch.Generator().manual_seed(zlib.crc32(name.encode()))
    q, do = rand_bf16((B, Hq, L, D), g), rand_bf16((B, Hq, L, D), g)
    k, v = rand_bf16((B, Hkv, S, D), g), rand_bf16((B, Hkv, S, D), g)
    _compare(_ids(cu_rows, S), q, k, v, do, s0, (p, SEED ^ zlib.crc32(name.encode()), 5), name)


def test_dropout_zero_is_the_plain_path(cuda_lib):
    wl = make_workload("tiny", 0)
    q, k, v, do = make_qkv_do(wl, device="cuda")
    ids = torch.from_numpy(_ids(wl.cu, wl.S)).cuda()
    seg, sid, nseg = A.segment_cu_seqlens(ids)
    plan = A.make_plan(seg, sid, nseg, wl.Hq, wl.Hkv, wl.L, 0)
    a = A.attn_forward(q, k, v, plan, 0, None, True)
    from packed_sequence_block_gb300 import _native as N
    out, lse = torch.empty_like(q), torch.empty_like(a[1])
    ws = torch.empty(N.bd_attn_fwd_planned_workspace_size(wl.B, wl.Hkv, wl.S, wl.D),
                     dtype=torch.uint8, device="cuda")
    N.bd_attn_fwd_dropout_planned(q, k, v, wl.B, wl.Hq, wl.Hkv, wl.L, wl.S, wl.D, 0,
                                  wl.D ** -0.5, True, plan, out, lse, 0.0, 123, 0, None, ws)
    assert torch.equal(out, a[0]) and torch.equal(lse, a[1])


def test_dropout_below_the_grain_is_the_plain_path(cuda_lib):
    """p < 2^-16 rounds to no dropout: bit-identical to the plain path."""
    wl = make_workload("tiny", 0)
    q, k, v, do = make_qkv_do(wl, device="cuda")
    ids = torch.from_numpy(_ids(wl.cu, wl.S)).cuda()
    r0 = gpu_forward_backward(q, k, v, do, ids)
    r1 = gpu_forward_backward(q, k, v, do, ids, dropout=(2.0 ** -17, 9, 0))
    for i in (0, 1, 3, 4):
        assert torch.equal(r0[i], r1[i])


def test_dropout_masks_follow_seed_and_offset(cuda_lib):
    wl = make_workload("tiny", 0)
    q, k, v, do = make_qkv_do(wl, device="cuda")
    ids = torch.from_numpy(_ids(wl.cu, wl.S)).cuda()
    r1 = gpu_forward_backward(q, k, v, do, ids, dropout=(0.3, 42, 0))
    r2 = gpu_forward_backward(q, k, v, do, ids, dropout=(0.3, 42, 0))
    for i in (0, 1, 3, 4):
        assert torch.equal(r1[i], r2[i])
    assert not torch.equal(gpu_forward_backward(q, k, v, do, ids, dropout=(0.3, 42, 1))[0], r1[0])
    assert not torch.equal(gpu_forward_backward(q, k, v, do, ids, dropout=(0.3, 43, 0))[0], r1[0])
    # lse is the undropped softmax's
    assert torch.equal(r1[1], gpu_forward_backward(q, k, v, do, ids)[1])


@pytest.mark.parametrize("p", [1.0, -0.1, float("nan")])
def test_dropout_rejects_bad_p(cuda_lib, p):
    wl = make_workload("tiny", 0)
    q, k, v, do = make_qkv_do(wl, device="cuda")
    ids = torch.from_numpy(_ids(wl.cu, wl.S)).cuda()
    with pytest.raises(ValueError):
        gpu_forward_backward(q, k, v, do, ids, dropout=(p, 1, 0))


def test_autograd_api_with_dropout(cuda_lib):
    from packed_sequence_block_gb300.attention import cp_blockdiag_sdpa
    S, Hq, Hkv, D, p, seed = 520, 4, 2, 128, 0.2, 77
    cu = [0, 200, 333, 520]
    g = torch.Generator().manual_seed(13)
    q, do = rand_bf16((1, Hq, S, D), g), rand_bf16((1, Hq, S, D), g)
    k, v = rand_bf16((1, Hkv, S, D), g), rand_bf16((1, Hkv, S, D), g)
    qa, ka, va = (t.clone().requires_grad_(True) for t in (q, k, v))
    out = cp_blockdiag_sdpa(qa, ka, va, dropout_p=p, enable_gqa=True, cu_seqlens=cu,
                            dropout_seed=seed, dropout_offset=2)
    out.backward(do)
    ids = _ids([cu], S)
    eo, el = orc.blockdiag_sdpa_forward(q, k, v, ids, 0, None, True, p, seed, 2)
    edq, edk, edv = orc.blockdiag_sdpa_backward(q, k, v, do, ids, 0, None, True, out=eo, lse=el,
                                                dropout_p=p, seed=seed, offset=2)
    assert_close("out", to64(out), eo)
    assert_close("dq", to64(qa.grad), edq)
    assert_close("dk", to64(ka.grad), edk)
    assert_close("dv", to64(va.grad), edv)


def test_dropout_lognormal8k_sampled(cuda_lib):
    """The 8192-token workload at full size with p = 0.1, checked on sampled rows
    and keys whose slices keep their planes and positions."""
    wl = make_workload("lognormal8k", 0)
    q, k, v, do = make_qkv_do(wl, device="cuda", generator_device="cuda")
    ids = torch.from_numpy(_ids(wl.cu, wl.S)).cuda()
    drop = (0.1, SEED, 1)
    out, lse, dq, dk, dv = gpu_forward_backward(q, k, v, do, ids, dropout=drop)
    rng = np.random.default_rng(8)
    sampled_checks(wl, q, k, v, do, out, lse, dq, dk, dv, 0, wl.L, 0, [0, 13, wl.Hq - 1], 5, rng,
                   dropout=drop)
