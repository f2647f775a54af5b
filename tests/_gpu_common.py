"""Shared helpers of the GPU parity tests (not collected as tests)."""
import numpy as np
import torch

from oracle import blockdiag as orc

# Tolerances of the parity bar (bf16 inputs/outputs, fp64 oracle):
# out, dq, dk, dv: max |err| <= 2e-2 beyond the rounding of a bf16 output
# (|got - exact| <= 2e-2 + 2^-8 |exact|; 2^-8 |x| bounds round-to-nearest
# bf16 error, which alone exceeds 2e-2 once |x| >= 8 and cannot be avoided by
# any bf16 result), and in the same reading mean |err| <= 2e-3 + 2^-9 mean
# |exact|, half the rounding bound on average (rounding the exact values to
# bf16 alone gives a mean error of ~1.9e-3 on a tensor whose mean |x| is 1.3);
# lse (fp32): max |err| <= 1e-3.
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
    mean_bar = mean_abs + 0.5 * BF16_ROUND * float(np.abs(exp).mean())
    assert ex <= max_abs and mn <= mean_bar, \
        f"{name}: max {mx:.3e} (beyond bf16 rounding {ex:.3e}) mean {mn:.3e} (bar {mean_bar:.3e})"
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


def gpu_forward_backward(q, k, v, do, doc_ids, seq_start=0, scale=None, enable_gqa=None,
                         dropout=None):
    """Run ids -> segments -> plan -> fwd -> bwd through the C ABI; return CUDA tensors.

    ``dropout`` is None or (p, seed, offset)."""
    from packed_sequence_block_gb300 import attention as A
    if enable_gqa is None:
        enable_gqa = q.shape[1] != k.shape[1]
    p, seed, offset = dropout if dropout is not None else (0.0, 0, 0)
    seg, sid, nseg = A.segment_cu_seqlens(doc_ids)
    plan = A.make_plan(seg, sid, nseg, q.shape[1], k.shape[1], q.shape[2], seq_start)
    out, lse, out16 = A.attn_forward(q, k, v, plan, seq_start, scale, enable_gqa,
                                      dropout_p=p, seed=seed, offset=offset)
    dq, dk, dv = A.attn_backward(q, k, v, out, lse, do, plan, seq_start, scale, enable_gqa,
                                 out16=out16, dropout_p=p, seed=seed, offset=offset)
    A.check_device_status(q.device)
    return out, lse, dq, dk, dv


def _sub_oracle_rows(q, k, v, do, b, hq_list, G, a, r0, r1, D, dropout=None):
    """Oracle on one document [a, r1) restricted to query rows [r0, r1) (all in the doc).

    With ``dropout`` = (p, seed, offset) the slice draws the whole problem's
    mask: its heads keep their planes b * Hq + h and its positions start at a."""
    qs = to64(q[b:b + 1, hq_list, r0:r1])
    dos = to64(do[b:b + 1, hq_list, r0:r1])
    kv_heads = sorted({h // G for h in hq_list})
    ks = to64(k[b:b + 1, kv_heads, a:r1])
    vs = to64(v[b:b + 1, kv_heads, a:r1])
    ids = np.ones((1, r1 - a), np.int32)
    Gs = len(hq_list) // len(kv_heads)
    kw = {}
    if dropout is not None:
        kw = dict(dropout_p=dropout[0], seed=dropout[1], offset=dropout[2],
                  mask_planes=[[b * q.shape[1] + h for h in hq_list]], mask_pos0=a)
    eo, el = orc.blockdiag_sdpa_forward(qs, ks, vs, ids, r0 - a, None, Gs > 1, **kw)
    edq, edk, edv = orc.blockdiag_sdpa_backward(qs, ks, vs, dos, ids, r0 - a, None, Gs > 1,
                                                out=eo, lse=el, **kw)
    return eo, el, edq, edk, edv


def sampled_checks(wl, q, k, v, do, out, lse, dq, dk, dv, s0, L, b, heads_fwd, group, rng,
                   dropout=None):
    """Rows near each document's start/end and tile boundaries; dk/dv of each doc's last keys."""
    G = wl.G
    cu = [int(x) for x in wl.cu[b]]
    last = cu[-1]
    for a, e in zip(cu[:-1], cu[1:]):
        lo, hi = max(a, s0), min(e, s0 + L)
        if lo >= hi:
            continue
        starts = {lo, max(lo, hi - 64), lo + (((hi - lo) // 2) // 128) * 128}
        starts.add(min(hi - 1, max(lo, int(rng.integers(lo, hi)))))
        for r0 in sorted(starts):
            r1 = min(hi, r0 + 64)
            if r1 <= r0:
                continue
            eo, el, edq, _, _ = _sub_oracle_rows(q, k, v, do, b, heads_fwd, G, a, r0, r1, wl.D, dropout)
            sl = slice(r0 - s0, r1 - s0)
            assert_close(f"out[{r0}:{r1}]", to64(out[b, heads_fwd, sl])[None], eo)
            assert_lse(f"lse[{r0}:{r1}]", to64(lse[b, heads_fwd, sl])[None], el)
            assert_close(f"dq[{r0}:{r1}]", to64(dq[b, heads_fwd, sl])[None], edq)
        # dk/dv of the last keys attended inside the interval: need only queries after them
        j0 = max(lo, hi - 128)
        heads = list(range(group * G, (group + 1) * G))
        _, _, _, edk, edv = _sub_oracle_rows(q, k, v, do, b, heads, G, a, j0, hi, wl.D, dropout)
        assert_close(f"dk[{j0}:{hi}]", to64(dk[b, group, j0:hi])[None, None], edk[:, :, j0 - a:])
        assert_close(f"dv[{j0}:{hi}]", to64(dv[b, group, j0:hi])[None, None], edv[:, :, j0 - a:])
    # padding rows and keys no query of the interval attends
    if last < s0 + L:
        pad = slice(max(last, s0) - s0, L)
        assert torch.all(out[b, :, pad] == 0) and torch.all(dq[b, :, pad] == 0)
        assert torch.all(torch.isneginf(lse[b, :, pad]))
    assert torch.all(dk[b, :, s0 + L:] == 0) and torch.all(dv[b, :, s0 + L:] == 0)
    assert torch.all(dk[b, :, last:] == 0) and torch.all(dv[b, :, last:] == 0)


def rand_bf16(shape, gen, device="cuda"):
    return torch.randn(shape, generator=gen, dtype=torch.float32).to(torch.bfloat16).to(device)
