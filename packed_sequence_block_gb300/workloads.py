"""Seeded synthetic workloads for block-diagonal causal attention over packed rows.

This module only draws numbers.  Document lengths come from
``numpy.random.default_rng(seed)``; q, k, v and the upstream gradient dO are
standard-normal fp32 draws from a ``torch.Generator`` seeded with ``seed`` and
rounded to bf16.  Nothing here computes any part of the attention method: the
CPU oracle and the CUDA path both consume what these functions return.

Five workloads are defined, with the shapes of the benchmark configurations:

``tiny``       1 row x 256 tokens, docs [37, 100, 1, 64, 54], Hq=4, Hkv=2, D=64
``lognormal8k`` 1 row x 8192 tokens, Hq=32, Hkv=8, D=128; lengths
               round(exp(N(ln 1024, 1.0))) clipped to [16, 8192], drawn until the
               next one would overflow the row; the rest of the row is padding
``shortdocs``  4 rows x 16384 tokens, Hq=Hkv=16, D=128; lengths uniform on
               [32, 512] per row, the last one cut so the row is exactly full
``interval131k`` 1 row x 131072 tokens, Hq=64, Hkv=8, D=128; 65536 tokens of
               lengths round(exp(N(ln 4096, 1.2))) clipped to [16, 65536], drawn
               until the next would overflow, then two 32768-token documents
               inserted at seeded places in the document order, tail padding;
               queries are 8 intervals of 16384 tokens at seq_start = k*16384
``causal64k``  2 rows x 65536 tokens, Hq=32, Hkv=4, D=64; one document of
               floor(0.95*65536) = 62259 tokens per row, then padding
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch


@dataclass
class Workload:
    """Shapes plus per-row document boundaries of one synthetic packed batch.

    ``cu[b]`` is row b's cumulative document boundary list (int32, first entry
    0, last entry <= S); positions at or past ``cu[b][-1]`` are padding.
    ``seq_starts`` lists the query intervals ``[s, s+L)`` that one step runs
    (a single ``[0]`` unless the row is split into intervals).
    """

    name: str
    B: int
    S: int
    L: int
    Hq: int
    Hkv: int
    D: int
    cu: list = field(default_factory=list)
    seq_starts: list = field(default_factory=lambda: [0])
    seed: int = 0

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    def cu_csr(self):
        """Rows' boundaries concatenated (int32) and the row pointer [B+1]."""
        flat = np.concatenate([np.asarray(c, np.int32) for c in self.cu]).astype(np.int32)
        row_ptr = np.zeros(self.B + 1, np.int32)
        row_ptr[1:] = np.cumsum([len(c) for c in self.cu])
        return flat, row_ptr

    def non_pad_tokens(self) -> int:
        """Number of non-padding query tokens over all rows and intervals."""
        total = 0
        for c in self.cu:
            last = int(c[-1])
            for s0 in self.seq_starts:
                total += max(0, min(last, s0 + self.L) - s0)
        return total


def _lognormal_docs(rng, median, sigma, lo, hi, budget):
    lens = []
    used = 0
    while True:
        x = int(np.clip(np.rint(np.exp(rng.normal(np.log(median), sigma))), lo, hi))
        if used + x > budget:
            break
        lens.append(x)
        used += x
    return lens


def _cu_from_lens(lens):
    cu = np.zeros(len(lens) + 1, np.int32)
    cu[1:] = np.cumsum(lens)
    return cu


def make_workload(name: str, seed: int = 0) -> Workload:
    """Build one of the named workloads with document lengths drawn from ``seed``."""
    rng = np.random.default_rng(seed)
    if name == "tiny":
        return Workload(name, 1, 256, 256, 4, 2, 64,
                        [_cu_from_lens([37, 100, 1, 64, 54])], [0], seed)
    if name == "lognormal8k":
        lens = _lognormal_docs(rng, 1024.0, 1.0, 16, 8192, 8192)
        return Workload(name, 1, 8192, 8192, 32, 8, 128, [_cu_from_lens(lens)], [0], seed)
    if name == "shortdocs":
        S = 16384
        cus = []
        for _ in range(4):
            lens = []
            used = 0
            while used < S:
                x = int(rng.integers(32, 512, endpoint=True))
                x = min(x, S - used)
                lens.append(x)
                used += x
            cus.append(_cu_from_lens(lens))
        return Workload(name, 4, S, S, 16, 16, 128, cus, [0], seed)
    if name == "interval131k":
        S = 131072
        lens = _lognormal_docs(rng, 4096.0, 1.2, 16, 65536, 65536)
        for _ in range(2):
            at = int(rng.integers(0, len(lens) + 1))
            lens.insert(at, 32768)
        return Workload(name, 1, S, 16384, 64, 8, 128, [_cu_from_lens(lens)],
                        [k * 16384 for k in range(8)], seed)
    if name == "causal64k":
        S = 65536
        n = int(0.95 * S)
        return Workload(name, 2, S, S, 32, 4, 64,
                        [_cu_from_lens([n]), _cu_from_lens([n])], [0], seed)
    raise ValueError(f"unknown workload {name!r}")


WORKLOADS = ("tiny", "lognormal8k", "shortdocs", "interval131k", "causal64k")


def random_cu(rng, S: int, max_docs: int = 8, pad_prob: float = 0.5,
              zero_len_prob: float = 0.15):
    """Random boundary list over S tokens: some zero-length docs, optional tail pad."""
    n = int(rng.integers(1, max_docs + 1))
    end = S if rng.random() > pad_prob else int(rng.integers(0, S + 1))
    cuts = np.sort(rng.integers(0, end + 1, size=n - 1)) if n > 1 else np.zeros(0, np.int64)
    cu = np.concatenate([[0], cuts, [end]]).astype(np.int32)
    for i in range(1, len(cu) - 1):
        if rng.random() < zero_len_prob:
            cu[i] = cu[i - 1]
    return np.maximum.accumulate(cu).astype(np.int32)


def make_tensors(B: int, H: int, T: int, D: int, seed: int, count: int,
                 device="cpu", generator_device=None):
    """``count`` bf16 tensors of shape [B, H, T, D], standard normal, drawn in order.

    The draw is fp32 ``torch.randn`` from one generator seeded with ``seed`` on
    ``generator_device`` (default: ``device``), then rounded to bf16.
    """
    gdev = torch.device(generator_device if generator_device is not None else device)
    g = torch.Generator(device=gdev)
    g.manual_seed(seed)
    out = []
    for _ in range(count):
        t = torch.randn((B, H, T, D), generator=g, device=gdev, dtype=torch.float32)
        out.append(t.to(torch.bfloat16).to(device))
    return out


def make_qkv_do(wl: Workload, seed: int | None = None, device="cpu", generator_device=None):
    """q [B,Hq,S,D], k, v [B,Hkv,S,D] and dO [B,Hq,S,D] for the whole row (bf16).

    q and dO cover every position of the row; an interval call takes the slice
    ``[:, :, s:s+L]``.  Draw order: q, k, v, dO.
    """
    seed = wl.seed if seed is None else seed
    gdev = torch.device(generator_device if generator_device is not None else device)
    g = torch.Generator(device=gdev)
    g.manual_seed(seed)

    def draw(H):
        t = torch.randn((wl.B, H, wl.S, wl.D), generator=g, device=gdev, dtype=torch.float32)
        return t.to(torch.bfloat16).to(device)

    q = draw(wl.Hq)
    k = draw(wl.Hkv)
    v = draw(wl.Hkv)
    do = draw(wl.Hq)
    return q, k, v, do
