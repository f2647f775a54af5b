"""Seeded random sweep of the single-call entry points against the oracle.

Each case draws its own shapes and document layout: 1-3 rows, up to 2,600
keys, a full row or an interval of queries (seq_start anywhere in the row),
1-3 K/V heads with 1-4 query heads each (GQA when more than one), D = 64 or
128, documents of random lengths (zero-length ones included) with optional
padding after the last one, and attention dropout in a third of the cases.
The mask is the per-document causal rule of cp_blockdiag_sdpa (page
"nemo_automodel.components.distributed.blockdiag_cp") on the ids of
doc_ids_from_cu_seqlens (page "nemo_automodel.components.models.glm5_next.cp").
out, lse, dq, dk and dv go through the C ABI (bd_attn_fwd / bd_attn_bwd and
their dropout forms) and are compared element by element with the fp64 oracle
under the bar the other parity tests use.  The layouts reach both forward work
orders (position order when every query block is short, longest first
otherwise) and documents that start and end anywhere inside a tile.
"""
import numpy as np
import pytest
import torch

from _gpu_common import assert_close, assert_lse, rand_bf16, to64
from oracle import blockdiag as orc
from packed_sequence_block_gb300 import attention as A

pytestmark = pytest.mark.gpu

N_CASES = 16


def _case(seed):
    rng = np.random.default_rng(1000 + seed)
    B = int(rng.integers(1, 4))
    S = int(rng.integers(1, 2601))
    if rng.random() < 0.5:
        s0, L = 0, S
    else:
        s0 = int(rng.integers(0, S))
        L = int(rng.integers(1, S - s0 + 1))
    Hkv = int(rng.integers(1, 4))
    G = int(rng.integers(1, 5))
    D = int(rng.choice([64, 128]))
    rows = []
    for _ in range(B):
        end = S if rng.random() < 0.6 else int(rng.integers(0, S + 1))  # padding after `end`
        cu, t = [0], 0
        while t < end:
            n = int(min(end - t, max(0, rng.lognormal(np.log(300), 1.2)) if rng.random() < 0.9 else 0))
            t += n
            cu.append(t)
        rows.append(cu)
    drop = (0.15, int(rng.integers(0, 2**63)), int(rng.integers(0, 2**31))) \
        if rng.random() < 1 / 3 else None
    return B, S, L, s0, Hkv * G, Hkv, D, rows, drop


@pytest.mark.parametrize("seed", range(N_CASES))
def test_random_single_call_matches_oracle(cuda_lib, seed):
    B, S, L, s0, Hq, Hkv, D, rows, drop = _case(seed)
    g = torch.Generator().manual_seed(seed)
    q, do = rand_bf16((B, Hq, L, D), g), rand_bf16((B, Hq, L, D), g)
    k, v = rand_bf16((B, Hkv, S, D), g), rand_bf16((B, Hkv, S, D), g)
    gqa = Hq != Hkv
    p, dseed, off = drop if drop is not None else (0.0, 0, 0)
    cu, rp = A.cu_csr(rows, "cuda")
    out, lse, ws = A.attn_forward_cu(q, k, v, cu, rp, s0, None, gqa, dropout_p=p, seed=dseed,
                                     offset=off)
    dq, dk, dv = A.attn_backward_cu(q, k, v, out, lse, do, cu, rp, ws, s0, None, gqa,
                                    dropout_p=p, seed=dseed, offset=off)
    A.check_device_status()
    ids = np.stack([orc.doc_ids_from_cu_seqlens(c, S) for c in rows])
    eo, el = orc.blockdiag_sdpa_forward(q, k, v, ids, s0, None, gqa, dropout_p=p, seed=dseed,
                                        offset=off)
    edq, edk, edv = orc.blockdiag_sdpa_backward(q, k, v, do, ids, s0, None, gqa, out=eo, lse=el,
                                                dropout_p=p, seed=dseed, offset=off)
    tag = f"case {seed} (B={B} S={S} L={L} s0={s0} Hq={Hq} Hkv={Hkv} D={D} p={p})"
    assert_close(f"{tag} out", to64(out), eo)
    assert_lse(f"{tag} lse", to64(lse), el)
    assert_close(f"{tag} dq", to64(dq), edq)
    assert_close(f"{tag} dk", to64(dk), edk)
    assert_close(f"{tag} dv", to64(dv), edv)
