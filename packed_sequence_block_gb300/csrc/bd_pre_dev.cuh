// Per-row terms of the backward pass, shared by the backward's own
// preprocess kernel and the single-call backward's first launch.
//
// The gradient of sum(out * dout) through the softmax of cp_blockdiag_sdpa
// (page "nemo_automodel.components.distributed.blockdiag_cp") needs, per query
// row i, Delta_i = <dO_i, o_i>; the main kernel also takes lse in log2 units.
// Both are written negated so that the main kernel adds them with paired fp32
// arithmetic.
#pragma once

#include "bd_ptx.cuh"

namespace bd {

constexpr float kLog2eF = 1.4426950408889634f;

// Threads per row of the per-row terms: each takes 32 of the row's D
// elements, as four 8-element pieces strided by the row's threads, so that
// its eight 16-byte loads are in flight together (one piece per load left
// the pass bound by load latency, not by HBM).
template <int D>
__host__ __device__ constexpr int pre_threads_per_row() { return D / 32; }

// Thread `tid` of planes * Lq * pre_threads_per_row<D>() takes its 32 elements
// of row (plane, i): their share of Delta (from the forward's fp16 O times
// o16_scale, the dropout scale 1 / (1 - p) that out carries and out16 does
// not, when out16 is given; else from the bf16 out), the zeroing of the same
// fp32 accumulator entries (when dqacc is given), and, in the row's first
// thread, -lse log2 e (-inf for rows that attend nothing) and -Delta.  Rows i
// in [L, Lq) get -inf and 0.  Whole warps must call it (the total is a
// multiple of 32); threads past the total return at once.
template <int D>
__device__ __forceinline__ void bwd_pre_rows(long long tid, const __nv_bfloat16* __restrict__ out,
                                             const __half* __restrict__ out16,
                                             float o16_scale,
                                             const __nv_bfloat16* __restrict__ dout,
                                             const float* __restrict__ lse, int planes, int L,
                                             int Lq, float* __restrict__ nlse2o,
                                             float* __restrict__ ndeltao,
                                             float* __restrict__ dqacc) {
  constexpr int TPR = pre_threads_per_row<D>();  // a power of two dividing 32
  constexpr int NP = 4;                          // pieces of 8 elements per thread
  static_assert(TPR * NP * 8 == D, "pieces must tile the row");
  if (tid >= (long long)planes * Lq * TPR) return;  // a multiple of 32: whole warps leave
  const long long rowg = tid / TPR;
  const int part = static_cast<int>(tid % TPR);
  const int plane = static_cast<int>(rowg / Lq);
  const int i = static_cast<int>(rowg % Lq);
  float acc = 0.f;
  if (i < L) {
    const size_t row = ((size_t)plane * L + i) * D;
    // piece j of this thread: elements [(j TPR + part) 8, + 8) of the row.
    // O is read only here (evict-first load); dO stays in L2 for the main
    // kernel that reads it next.
    uint4 d4[NP], o4[NP];
    const bool hp = out16 != nullptr;
#pragma unroll
    for (int j = 0; j < NP; ++j) {
      const size_t off = row + (size_t)(j * TPR + part) * 8;
      d4[j] = *reinterpret_cast<const uint4*>(dout + off);
      o4[j] = hp ? __ldcs(reinterpret_cast<const uint4*>(out16 + off))
                 : __ldcs(reinterpret_cast<const uint4*>(out + off));
    }
#pragma unroll
    for (int j = 0; j < NP; ++j) {
      const __nv_bfloat162* d2 = reinterpret_cast<const __nv_bfloat162*>(&d4[j]);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 a = hp ? __half22float2(reinterpret_cast<const __half2*>(&o4[j])[e])
                            : __bfloat1622float2(reinterpret_cast<const __nv_bfloat162*>(&o4[j])[e]);
        const float2 b = __bfloat1622float2(d2[e]);
        acc = fmaf(a.x, b.x, acc);
        acc = fmaf(a.y, b.y, acc);
      }
    }
    if (dqacc != nullptr) {
#pragma unroll
      for (int j = 0; j < NP; ++j) {
        float4* z = reinterpret_cast<float4*>(dqacc + row + (size_t)(j * TPR + part) * 8);
        z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
        z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
  }
  // every lane of the warp takes part in the shuffles (rows past L add 0)
#pragma unroll
  for (int o = TPR / 2; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o, TPR);
  if (part == 0) {
    float nl2 = -INFINITY, ndl = 0.f;
    if (i < L) {
      const float x = lse[(size_t)plane * L + i];
      if (x != -INFINITY) {
        nl2 = -(x * kLog2eF);
        ndl = out16 != nullptr ? -(acc * o16_scale) : -acc;
      }
    }
    nlse2o[(size_t)plane * Lq + i] = nl2;
    ndeltao[(size_t)plane * Lq + i] = ndl;
  }
}

}  // namespace bd
