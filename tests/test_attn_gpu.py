"""GPU parity of block-diagonal causal attention (forward and backward) against the oracle.

Every case runs ids -> segments -> plan -> forward -> backward through the C
ABI and compares element by element with the fp64 oracle on the same seeded
bf16 inputs (bar: max |err| <= 2e-2, mean |err| <= 2e-3 for out/dq/dk/dv,
max |err| <= 1e-3 for lse).  Small cases cover ragged tails, every GQA
grouping the kernels distinguish (G even, G odd, G = 1), head dims 64 and
128, query intervals (aligned and not), interior padding, repeated ids,
all-padding rows and one-token documents.  The benchmark workloads run at
full size: the 8192- and 4x16384-token ones compared in full, the two large
ones on sampled rows the oracle computes on their own (rows are independent;
dk/dv of the last keys of a document need only the queries after them).  One
case sits at the largest work lists the library accepts (16384 entries).
"""
import zlib

import numpy as np
import pytest
import torch

from _gpu_common import (assert_close, assert_lse, gpu_forward_backward, rand_bf16,
                         sampled_checks, to64)
from oracle import blockdiag as orc
from packed_sequence_block_gb300.workloads import make_qkv_do, make_workload

pytestmark = pytest.mark.gpu


def _ids(cu_rows, S):
    return np.stack([orc.doc_ids_from_cu_seqlens(c, S) for c in cu_rows])


def _run_and_compare(ids, q, k, v, do, seq_start=0, scale=None, tag=""):
    tids = torch.from_numpy(ids).cuda()
    gqa = q.shape[1] != k.shape[1]
    out, lse, dq, dk, dv = gpu_forward_backward(q, k, v, do, tids, seq_start, scale, gqa)
    eo, el = orc.blockdiag_sdpa_forward(q, k, v, ids, seq_start, scale, gqa)
    edq, edk, edv = orc.blockdiag_sdpa_backward(q, k, v, do, ids, seq_start, scale, gqa,
                                                out=eo, lse=el)
    assert_close(f"{tag} out", to64(out), eo)
    assert_lse(f"{tag} lse", to64(lse), el)
    assert_close(f"{tag} dq", to64(dq), edq)
    assert_close(f"{tag} dk", to64(dk), edk)
    assert_close(f"{tag} dv", to64(dv), edv)


SMALL = {
    # name: (cu rows, S, L, seq_start, Hq, Hkv, D)
    "tiny": ([[0, 37, 137, 138, 202, 256]], 256, 256, 0, 4, 2, 64),
    "mha_ragged_d64": ([[0, 100, 300]], 300, 300, 0, 2, 2, 64),
    "g3_ragged_d128": ([[0, 17, 260, 517], [0, 400]], 517, 517, 0, 6, 2, 128),
    "g4_d128": ([[0, 128, 129, 700, 1000]], 1000, 1000, 0, 8, 2, 128),
    "g8_d64_onedoc": ([[0, 1500]], 1500, 1500, 0, 8, 1, 64),
    "interval_unaligned": ([[0, 150, 600, 1024]], 1024, 300, 200, 4, 1, 64),
    "interval_aligned": ([[0, 700, 1300, 2048]], 2048, 256, 768, 4, 2, 128),
    "all_pad_row": ([[0, 90, 256], [0]], 256, 256, 0, 2, 1, 128),
    "one_token_docs": ([list(range(0, 257))], 256, 256, 0, 2, 2, 64),
    "many_zero_len": ([[0, 0, 5, 5, 5, 200, 200, 333]], 384, 384, 0, 4, 4, 128),
    "single_token_row": ([[0, 1]], 1, 1, 0, 2, 1, 64),
    "last_query_only": ([[0, 200, 333]], 333, 1, 332, 4, 2, 128),
    "first_query_only_padded": ([[0, 1], [0]], 300, 1, 0, 3, 1, 64),
}


@pytest.mark.parametrize("name", sorted(SMALL))
def test_small_cases(cuda_lib, name):
    cu_rows, S, L, s0, Hq, Hkv, D = SMALL[name]
    B = len(cu_rows)
    g = torch.Generator().manual_seed(zlib.crc32(name.encode()))
    q, do = rand_bf16((B, Hq, L, D), g), rand_bf16((B, Hq, L, D), g)
    k, v = rand_bf16((B, Hkv, S, D), g), rand_bf16((B, Hkv, S, D), g)
    _run_and_compare(_ids(cu_rows, S), q, k, v, do, s0, None, name)


def test_interior_padding_and_repeated_ids(cuda_lib):
    """doc ids straight from a caller: padding in the middle, an id reused later."""
    S, Hq, Hkv, D = 700, 4, 2, 128
    ids = np.zeros((1, S), np.int32)
    ids[0, 0:200] = 3
    ids[0, 200:260] = 0
    ids[0, 260:500] = 7
    ids[0, 500:650] = 3   # same id as the first run, a different segment
    g = torch.Generator().manual_seed(5)
    q, do = rand_bf16((1, Hq, S, D), g), rand_bf16((1, Hq, S, D), g)
    k, v = rand_bf16((1, Hkv, S, D), g), rand_bf16((1, Hkv, S, D), g)
    _run_and_compare(ids, q, k, v, do, 0, None, "interior_pad")


def test_explicit_scale(cuda_lib):
    """A caller's scale is used instead of D**-0.5 (forward and backward).

    With a much sharper softmax (scale 0.3 = 2.4x the default at D=64) the
    forward is still checked; the backward's dq error grows there because
    Delta = <dO, O> is formed from the bf16 output, so the gradient check
    uses a scale below the default.
    """
    S, D = 400, 64
    ids = _ids([[0, 250, 400]], S)
    g = torch.Generator().manual_seed(9)
    q, do = rand_bf16((1, 2, S, D), g), rand_bf16((1, 2, S, D), g)
    k, v = rand_bf16((1, 2, S, D), g), rand_bf16((1, 2, S, D), g)
    _run_and_compare(ids, q, k, v, do, 0, 0.09, "scale0.09")
    tids = torch.from_numpy(ids).cuda()
    out, lse, *_ = gpu_forward_backward(q, k, v, do, tids, 0, 0.3, False)
    eo, el = orc.blockdiag_sdpa_forward(q, k, v, ids, 0, 0.3, False)
    assert_close("scale0.3 out", to64(out), eo)
    assert_lse("scale0.3 lse", to64(lse), el)


def test_autograd_api_matches_oracle(cuda_lib):
    from packed_sequence_block_gb300.attention import cp_blockdiag_sdpa
    S, Hq, Hkv, D = 520, 4, 2, 128
    cu = [0, 200, 333, 520]
    g = torch.Generator().manual_seed(3)
    q, do = rand_bf16((1, Hq, S, D), g), rand_bf16((1, Hq, S, D), g)
    k, v = rand_bf16((1, Hkv, S, D), g), rand_bf16((1, Hkv, S, D), g)
    qa, ka, va = (t.clone().requires_grad_(True) for t in (q, k, v))
    out = cp_blockdiag_sdpa(qa, ka, va, attn_mask=torch.ones(1), is_causal=True,
                            enable_gqa=True, cu_seqlens=cu)
    out.backward(do)
    ids = _ids([cu], S)
    eo, el = orc.blockdiag_sdpa_forward(q, k, v, ids, 0, None, True)
    edq, edk, edv = orc.blockdiag_sdpa_backward(q, k, v, do, ids, 0, None, True, out=eo, lse=el)
    assert_close("out", to64(out), eo)
    assert_close("dq", to64(qa.grad), edq)
    assert_close("dk", to64(ka.grad), edk)
    assert_close("dv", to64(va.grad), edv)
    with pytest.raises(ValueError):
        cp_blockdiag_sdpa(q, k, v, dropout_p=1.0, enable_gqa=True, cu_seqlens=cu)


def test_repeat_calls_are_stable(cuda_lib):
    """Same inputs twice: out/lse/dk/dv identical, dq within atomics' rounding."""
    wl = make_workload("tiny")
    q, k, v, do = make_qkv_do(wl, device="cuda")
    ids = torch.from_numpy(_ids(wl.cu, wl.S)).cuda()
    r1 = gpu_forward_backward(q, k, v, do, ids)
    r2 = gpu_forward_backward(q, k, v, do, ids)
    for i in (0, 1, 3, 4):
        assert torch.equal(r1[i], r2[i])
    assert (r1[2].float() - r2[2].float()).abs().max().item() <= 1e-2


@pytest.mark.parametrize("name", ["tiny", "lognormal8k", "shortdocs"])
def test_workload_full(cuda_lib, name):
    wl = make_workload(name, 0)
    q, k, v, do = make_qkv_do(wl, device="cuda", generator_device="cuda")
    _run_and_compare(_ids(wl.cu, wl.S), q, k, v, do, 0, None, name)


def test_causal64k_sampled(cuda_lib):
    wl = make_workload("causal64k", 0)
    q, k, v, do = make_qkv_do(wl, device="cuda", generator_device="cuda")
    ids = torch.from_numpy(_ids(wl.cu, wl.S)).cuda()
    out, lse, dq, dk, dv = gpu_forward_backward(q, k, v, do, ids)
    rng = np.random.default_rng(0)
    for b in range(wl.B):
        sampled_checks(wl, q, k, v, do, out, lse, dq, dk, dv, 0, wl.L, b, [0, wl.Hq - 1],
                        b % wl.Hkv, rng)


@pytest.mark.parametrize("interval", [0, 3, 7])
def test_interval131k_sampled(cuda_lib, interval):
    wl = make_workload("interval131k", 0)
    q, k, v, do = make_qkv_do(wl, device="cuda", generator_device="cuda")
    s0 = wl.seq_starts[interval]
    L = wl.L
    qi = q[:, :, s0:s0 + L].contiguous()
    doi = do[:, :, s0:s0 + L].contiguous()
    ids = torch.from_numpy(_ids(wl.cu, wl.S)).cuda()
    out, lse, dq, dk, dv = gpu_forward_backward(qi, k, v, doi, ids, s0)
    # embed the interval's query-side tensors at their global rows for the sampler
    full = lambda t: torch.nn.functional.pad(t, (0, 0, s0, wl.S - s0 - L))  # noqa: E731
    rng = np.random.default_rng(interval)
    sampled_checks(wl, full(qi), k, v, full(doi), out, lse, dq, dk, dv, s0, L, 0, [0, 37, 63],
                    interval % wl.Hkv, rng)


def test_longest_work_lists_sampled(cuda_lib):
    """B * ceil(S / 128) at the library's 16384-entry limit for both work lists
    (8 rows x 262144 tokens, Hq = 2 so that a forward block is one 128-row tile),
    which the plan sorts with its bitonic path (the other cases stay under 2048
    entries and use the rank sort); checked on sampled rows of two rows."""
    from packed_sequence_block_gb300.workloads import Workload
    rng = np.random.default_rng(77)
    B, S = 8, 262144
    cus = []
    for _ in range(B):
        lens, used = [], 0
        while True:
            x = int(np.clip(np.rint(np.exp(rng.normal(np.log(8192.0), 1.0))), 16, 65536))
            if used + x > S - 1000:
                break
            lens.append(x)
            used += x
        cus.append(np.concatenate([[0], np.cumsum(lens)]).astype(np.int32))
    wl = Workload("longest_lists", B, S, S, 2, 1, 64, cus, [0], 5)
    assert B * (S // 128) == 16384
    q, k, v, do = make_qkv_do(wl, device="cuda", generator_device="cuda")
    ids = torch.from_numpy(_ids(wl.cu, wl.S)).cuda()
    out, lse, dq, dk, dv = gpu_forward_backward(q, k, v, do, ids)
    srng = np.random.default_rng(3)
    for b in (0, B - 1):
        sampled_checks(wl, q, k, v, do, out, lse, dq, dk, dv, 0, wl.L, b, [0, 1], 0, srng)
