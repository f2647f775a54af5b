"""Seeded random sweep of the planned path (ids -> segments -> plan -> kernels)
against the oracle, on document-id rows that boundaries cannot express.

Each row is a sequence of runs of ids drawn at random: padding runs (id 0)
anywhere, including first and between documents, and ids that repeat after a
gap or after another document.  The mask is cp_blockdiag_sdpa's (page
"nemo_automodel.components.distributed.blockdiag_cp"): a query attends the keys
at or before it inside its own segment, a maximal run of equal non-zero ids
(segment_cu_seqlens, page "nemo_automodel.components.models.glm5_next.cp"), so
a repeated id after a gap starts a new document.  Shapes, intervals, GQA, D
and dropout are drawn as in the single-call sweep; out, lse, dq, dk and dv are
compared element by element with the fp64 oracle.
"""
import numpy as np
import pytest
import torch

from _gpu_common import assert_close, assert_lse, gpu_forward_backward, rand_bf16, to64
from oracle import blockdiag as orc

pytestmark = pytest.mark.gpu

N_CASES = 8


def _case(seed):
    rng = np.random.default_rng(5000 + seed)
    B = int(rng.integers(1, 4))
    S = int(rng.integers(1, 1801))
    if rng.random() < 0.5:
        s0, L = 0, S
    else:
        s0 = int(rng.integers(0, S))
        L = int(rng.integers(1, S - s0 + 1))
    Hkv = int(rng.integers(1, 4))
    G = int(rng.integers(1, 5))
    D = int(rng.choice([64, 128]))
    ids = np.zeros((B, S), np.int32)
    for b in range(B):
        t, nxt = 0, 1
        while t < S:
            n = int(min(S - t, max(1, rng.lognormal(np.log(150), 1.1))))
            u = rng.random()
            if u < 0.25:
                v = 0                                  # padding run
            elif u < 0.4 and nxt > 1:
                v = int(rng.integers(1, nxt))          # an id seen before
            else:
                v, nxt = nxt, nxt + 1
            ids[b, t:t + n] = v
            t += n
    drop = (0.2, int(rng.integers(0, 2**63)), int(rng.integers(0, 2**31))) \
        if rng.random() < 1 / 3 else None
    return B, S, L, s0, Hkv * G, Hkv, D, ids, drop


@pytest.mark.parametrize("seed", range(N_CASES))
def test_random_ids_planned_matches_oracle(cuda_lib, seed):
    B, S, L, s0, Hq, Hkv, D, ids, drop = _case(seed)
    g = torch.Generator().manual_seed(100 + seed)
    q, do = rand_bf16((B, Hq, L, D), g), rand_bf16((B, Hq, L, D), g)
    k, v = rand_bf16((B, Hkv, S, D), g), rand_bf16((B, Hkv, S, D), g)
    gqa = Hq != Hkv
    out, lse, dq, dk, dv = gpu_forward_backward(q, k, v, do, torch.from_numpy(ids).cuda(), s0,
                                                dropout=drop)
    p, dseed, off = drop if drop is not None else (0.0, 0, 0)
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
