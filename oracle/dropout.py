"""Oracle for attention dropout: the keep mask and its counter-based generator.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
legs of ``bench.py`` may import or run this module; the product path never
does, and this module imports nothing from the product package.

What it follows:

* Page "nemo_automodel.components.distributed.blockdiag_cp",
  ``cp_blockdiag_sdpa(..., dropout_p: float = 0.0, ...)``: a drop-in for torch
  scaled_dot_product_attention, where dropout_p is the dropout probability.
  Reading (SDPA's convention): dropout acts on the normalised attention
  weights P; a kept weight is scaled by 1 / (1 - p), a dropped one is 0; the
  returned log-sum-exp is the softmax's, before dropout.
* The random bits: Philox4x32-10, the counter-based generator of Salmon,
  Moraes, Dror and Shaw, "Parallel random numbers: as easy as 1, 2, 3"
  (SC'11): ten rounds on a 128-bit counter (four 32-bit words) under a 64-bit
  key (two words); a round multiplies counter words 0 and 2 by 0xD2511F53 and
  0xCD9E8D57, and maps (c0, c1, c2, c3) to (hi(M1 c2) ^ c1 ^ k0, lo(M1 c2),
  hi(M0 c0) ^ c3 ^ k1, lo(M0 c0)); between rounds the key words grow by
  0x9E3779B9 and 0xBB67AE85.  The same generator is written independently on
  the device from that definition.

Reading for the mask (no page fixes one): each weight draws a 16-bit value.
Element (plane = b Hq + h, query at global position t, key at position j)
uses counter (j >> 3, t, plane, offset) under key (seed & 0xffffffff,
seed >> 32); of the four output words, word (j & 7) >> 1 holds its value, in
the low 16 bits for even j and the high 16 bits for odd j.  It is kept iff
that value >= floor(p * 2**16).  The drop probability is therefore p rounded
down to a multiple of 2**-16, p' = floor(p * 2**16) / 2**16, and kept weights
are scaled by 1 / (1 - p'), which keeps the expectation exact.  The query's
global position (not its local row) enters the counter, so a row split into
query intervals draws the same mask as the whole row.

Pins: the generator's words equal those of an independent implementation,
cuRAND's device Philox4_32_10 (tests/test_oracle_philox_gpu.py, run on a
GPU), for random seeds and counters; on the CPU it is held by properties
(bijectivity, uniform words, the drop rate, independent neighbouring keys).
The dropout arithmetic is pinned by exact reductions (p = 0, a dense
restatement, the expectation over masks, finite differences with the mask
fixed).
"""
from __future__ import annotations

import numpy as np

_M0, _M1 = np.uint64(0xD2511F53), np.uint64(0xCD9E8D57)
_W0, _W1 = 0x9E3779B9, 0xBB67AE85
_MASK32 = np.uint64(0xFFFFFFFF)


def philox4x32_10(c0, c1, c2, c3, seed: int):
    """Philox4x32-10 on arrays of counter words (broadcast together), 64-bit seed."""
    c = [np.asarray(x, dtype=np.uint64) & _MASK32 for x in (c0, c1, c2, c3)]
    c = np.broadcast_arrays(*c)
    c0, c1, c2, c3 = [x.copy() for x in c]
    k0, k1 = seed & 0xFFFFFFFF, (seed >> 32) & 0xFFFFFFFF
    for _ in range(10):
        p0 = c0 * _M0
        p1 = c2 * _M1
        hi0, lo0 = p0 >> np.uint64(32), p0 & _MASK32
        hi1, lo1 = p1 >> np.uint64(32), p1 & _MASK32
        c0, c1, c2, c3 = (hi1 ^ c1 ^ np.uint64(k0), lo1, hi0 ^ c3 ^ np.uint64(k1), lo0)
        k0 = (k0 + _W0) & 0xFFFFFFFF
        k1 = (k1 + _W1) & 0xFFFFFFFF
    return tuple(x.astype(np.uint32) for x in (c0, c1, c2, c3))


def drop_threshold(p: float) -> int:
    """16-bit values below floor(p * 2**16) drop their element (p in [0, 1))."""
    if not 0.0 <= p < 1.0:
        raise ValueError("dropout_p must lie in [0, 1)")
    return int(np.floor(float(p) * 65536.0))


def keep_scale(p: float) -> float:
    """1 / (1 - p') for the drop probability p' = drop_threshold(p) / 2**16."""
    return 1.0 / (1.0 - drop_threshold(p) / 65536.0)


def keep_mask(plane: int, t, j, seed: int, offset: int, p: float) -> np.ndarray:
    """Boolean keep mask [len(t), len(j)] of query positions t against key positions j."""
    t = np.asarray(t, dtype=np.int64)[:, None]
    j = np.asarray(j, dtype=np.int64)[None, :]
    words = philox4x32_10(j >> 3, t, np.int64(plane), np.int64(offset), seed)
    shape = np.broadcast_shapes(t.shape, j.shape)
    w = np.choose(np.broadcast_to((j & 7) >> 1, shape), words)
    half = (w >> np.broadcast_to(((j & 1) * 16).astype(np.uint32), shape)) & np.uint32(0xFFFF)
    return half >= np.uint32(drop_threshold(p)) if p > 0.0 else np.ones(half.shape, bool)
