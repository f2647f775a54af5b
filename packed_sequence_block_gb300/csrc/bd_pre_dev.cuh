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

// Thread `tid` of planes * Lq * (D / 8) takes 8 elements of row (plane, i):
// their share of Delta (from out + out_lo when out_lo is given), the zeroing
// of the same 8 fp32 accumulator entries (when dqacc is given), and, in the
// row's first thread,
// -lse log2 e (-inf for rows that attend nothing) and -Delta.  Rows i in
// [L, Lq) get -inf and 0.  Whole warps must call it (the total is a multiple
// of 32); threads past the total return at once.
template <int D>
__device__ __forceinline__ void bwd_pre_rows(long long tid, const __nv_bfloat16* __restrict__ out,
                                             const __nv_bfloat16* __restrict__ out_lo,
                                             const __nv_bfloat16* __restrict__ dout,
                                             const float* __restrict__ lse, int planes, int L,
                                             int Lq, float* __restrict__ nlse2o,
                                             float* __restrict__ ndeltao,
                                             float* __restrict__ dqacc) {
  constexpr int TPR = D / 8;  // threads per row (a power of two dividing 32)
  if (tid >= (long long)planes * Lq * TPR) return;  // a multiple of 32: whole warps leave
  const long long rowg = tid / TPR;
  const int part = static_cast<int>(tid % TPR);
  const int plane = static_cast<int>(rowg / Lq);
  const int i = static_cast<int>(rowg % Lq);
  float acc = 0.f;
  if (i < L) {
    const size_t off = ((size_t)plane * L + i) * D + part * 8;
    const uint4 o4 = *reinterpret_cast<const uint4*>(out + off);
    const uint4 d4 = *reinterpret_cast<const uint4*>(dout + off);
    const uint4 l4 = out_lo != nullptr ? *reinterpret_cast<const uint4*>(out_lo + off)
                                       : make_uint4(0, 0, 0, 0);
    const __nv_bfloat162* o2 = reinterpret_cast<const __nv_bfloat162*>(&o4);
    const __nv_bfloat162* l2v = reinterpret_cast<const __nv_bfloat162*>(&l4);
    const __nv_bfloat162* d2 = reinterpret_cast<const __nv_bfloat162*>(&d4);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 a = __bfloat1622float2(o2[j]);
      const float2 r = __bfloat1622float2(l2v[j]);
      const float2 b = __bfloat1622float2(d2[j]);
      acc = fmaf(a.x + r.x, b.x, acc);
      acc = fmaf(a.y + r.y, b.y, acc);
    }
    if (dqacc != nullptr) {
      float4* z = reinterpret_cast<float4*>(dqacc + off);
      z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
      z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
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
        ndl = -acc;
      }
    }
    nlse2o[(size_t)plane * Lq + i] = nl2;
    ndeltao[(size_t)plane * Lq + i] = ndl;
  }
}

}  // namespace bd
