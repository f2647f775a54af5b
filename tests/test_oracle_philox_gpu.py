"""Pins the oracle's Philox4x32-10 to an independent implementation: cuRAND's
device generator (curandStatePhilox4_32_10_t).

curand_init(seed, subsequence, 0, &state) followed by curand4(&state) returns
the generator's four words at counter (0, 0, subsequence mod 2^32,
subsequence >> 32) under key (seed mod 2^32, seed >> 32).  Agreement on random
seeds and subsequences pins the round function and the key schedule
(Salmon et al., SC'11) that the oracle writes out, and with them the exact
stream the dropout mask draws from.  cuRAND serves this test only; neither
the library nor the oracle uses it.
"""
import ctypes
import os
import shutil
import subprocess
import tempfile

import numpy as np
import pytest
import torch

from oracle import dropout as dro

pytestmark = pytest.mark.gpu

_SRC = r"""
#include <curand_kernel.h>
#include <stdint.h>
__global__ void words(unsigned long long seed, const unsigned long long* sub, uint4* out, int n) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  curandStatePhilox4_32_10_t st;
  curand_init(seed, sub[i], 0, &st);
  out[i] = curand4(&st);
}
extern "C" int philox_words(unsigned long long seed, const void* sub, void* out, int n) {
  words<<<(n + 127) / 128, 128>>>(seed, static_cast<const unsigned long long*>(sub),
                                  static_cast<uint4*>(out), n);
  return static_cast<int>(cudaDeviceSynchronize());
}
"""


@pytest.fixture(scope="module")
def curand_words():
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    d = tempfile.mkdtemp()
    src, so = os.path.join(d, "w.cu"), os.path.join(d, "w.so")
    open(src, "w").write(_SRC)
    subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-shared",
                    "-Xcompiler", "-fPIC", src, "-o", so], check=True)
    lib = ctypes.CDLL(so)
    lib.philox_words.argtypes = [ctypes.c_ulonglong, ctypes.c_void_p, ctypes.c_void_p,
                                 ctypes.c_int]

    def run(seed, subs):
        sub = torch.tensor(np.asarray(subs, np.uint64).view(np.int64), device="cuda")
        out = torch.empty((len(subs), 4), dtype=torch.int32, device="cuda")
        assert lib.philox_words(seed, sub.data_ptr(), out.data_ptr(), len(subs)) == 0
        return out.cpu().numpy().view(np.uint32)
    return run


@pytest.mark.parametrize("seed", [0, 1, 0x9E3779B97F4A7C15, 0xFFFFFFFF00000001, 20240607])
def test_oracle_philox_matches_curand(curand_words, seed):
    rng = np.random.default_rng(seed % (1 << 32))
    subs = np.concatenate([np.arange(64, dtype=np.uint64),
                           rng.integers(0, 1 << 63, 448, dtype=np.uint64),
                           np.array([(1 << 32) - 1, 1 << 32, (1 << 64) - 1], dtype=np.uint64)])
    got = curand_words(seed, subs)
    w = dro.philox4x32_10(0, 0, subs & np.uint64(0xFFFFFFFF), subs >> np.uint64(32), seed)
    want = np.stack([x.astype(np.uint32) for x in w], axis=1)
    np.testing.assert_array_equal(want, got)
