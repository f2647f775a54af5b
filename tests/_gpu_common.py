"""Shared helpers of the GPU parity tests (not collected as tests)."""
import numpy as np
import torch

# Tolerances of the parity bar (bf16 inputs/outputs, fp64 oracle):
# out, dq, dk, dv: max |err| <= 2e-2 beyond the rounding of a bf16 output
# (|got - exact| <= 2e-2 + 2^-8 |exact|; 2^-8 |x| bounds round-to-nearest
# bf16 error, which alone exceeds 2e-2 once |x| >= 8 and cannot be avoided by
# any bf16 result), and mean |err| <= 2e-3; lse (fp32): max |err| <= 1e-3.
MAX_ABS = 2e-2
MEAN_ABS = 2e-3
LSE_ABS = 1e-3
BF16_ROUND = 2.0 ** -8


def to64(t):
    return t.detach().to("cpu", torch.float64).numpy()


def assert_close(name, got, exp, max_abs=MAX_ABS, mean_abs=MEAN_ABS):
    got = np.asarray(got, np.float64)
    exp = np.asarray(exp, np.float64)
    assert got.shape == exp.shape, f"{name}: shape {got.shape} vs {exp.shape}"
    assert np.all(np.isfinite(got)), f"{name}: non-finite values"
    err = np.abs(got - exp)
    if not err.size:
        return 0.0, 0.0
    excess = np.maximum(0.0, err - BF16_ROUND * np.abs(exp))
    mx, mn, ex = float(err.max()), float(err.mean()), float(excess.max())
    assert ex <= max_abs and mn <= mean_abs, \
        f"{name}: max {mx:.3e} (beyond bf16 rounding {ex:.3e}) mean {mn:.3e}"
    return mx, mn


def assert_lse(name, got, exp, tol=LSE_ABS):
    got = np.asarray(got, np.float64)
    exp = np.asarray(exp, np.float64)
    assert got.shape == exp.shape
    inf_e = np.isneginf(exp)
    assert np.array_equal(np.isneginf(got), inf_e), f"{name}: -inf pattern differs"
    fin = ~inf_e
    if fin.any():
        err = float(np.abs(got[fin] - exp[fin]).max())
        assert err <= tol, f"{name}: max {err:.3e}"


def gpu_forward_backward(q, k, v, do, doc_ids, seq_start=0, scale=None, enable_gqa=None):
    """Run ids -> segments -> plan -> fwd -> bwd through the C ABI; return CUDA tensors."""
    from packed_sequence_block_gb300 import attention as A
    if enable_gqa is None:
        enable_gqa = q.shape[1] != k.shape[1]
    seg, sid, nseg = A.segment_cu_seqlens(doc_ids)
    plan = A.make_plan(seg, sid, nseg, q.shape[1], k.shape[1], q.shape[2], seq_start)
    out, lse, out_lo = A.attn_forward(q, k, v, plan, seq_start, scale, enable_gqa)
    dq, dk, dv = A.attn_backward(q, k, v, out, lse, do, plan, seq_start, scale, enable_gqa,
                                 out_lo=out_lo)
    A.check_device_status(q.device)
    return out, lse, dq, dk, dv


def rand_bf16(shape, gen, device="cuda"):
    return torch.randn(shape, generator=gen, dtype=torch.float32).to(torch.bfloat16).to(device)
