// First launches of the single-call forward and backward (bd_attn_fwd and
// bd_attn_bwd, which take cumulative document boundaries).  Each is one
// launch whose block 0 builds the attention plan from the boundaries (the
// mask bounds of every row and the ordered work lists, see
// bd_plan_dev.cuh) while the other blocks do the pass over HBM that the call
// needs anyway: the fp16 copy of v and the plan's per-position mask bounds
// before the forward, the per-row terms before the backward.
#include "bd_plan_dev.cuh"
#include "bd_pre_dev.cuh"

namespace bd {

namespace {

constexpr int kPrepFwdThreads = 1024;
constexpr int kPrepBwdThreads = 256;

__device__ __forceinline__ void plan_block(const int32_t* cu, const int32_t* row_ptr,
                                           const PlanPtrs& pp, int32_t* status, bool write_rows) {
  extern __shared__ unsigned long long prep_smem[];
  const int nf = pp.B * pp.NQB, nb = pp.B * pp.NKT;
  int np = 1;
  while (np < max(nf, nb)) np <<= 1;
  const int bad_words = (pp.B + 31) / 32;
  // as plan_cta_smem lays it out: keys, row bits, boundary cache
  const int nkeys = (nf <= kRankSortMax && nb <= kRankSortMax) ? max(np, nf + nb) : np;
  uint32_t* bad = reinterpret_cast<uint32_t*>(prep_smem + nkeys);
  int32_t* cache = reinterpret_cast<int32_t*>(bad + bad_words);
  build_plan_cta(cu, row_ptr, pp, status, prep_smem, bad, bad_words, cache, write_rows);
}

// The header records the forward of these inputs (flags aside).
__device__ __forceinline__ bool same_tag(const WsTag* h, const WsTag& e) {
  return h->magic == e.magic && h->B == e.B && h->Hq == e.Hq && h->Hkv == e.Hkv &&
         h->L == e.L && h->S == e.S && h->D == e.D && h->seq_start == e.seq_start &&
         h->out == e.out && h->lse == e.lse && h->cu == e.cu && h->row_ptr == e.row_ptr;
}

__global__ void __launch_bounds__(kPrepFwdThreads) prep_fwd_kernel(
    const int32_t* __restrict__ cu, const int32_t* __restrict__ row_ptr, const PlanPtrs pp,
    const WsTag tag, WsTag* hdr, const uint4* __restrict__ v, uint4* __restrict__ v16,
    long long n8, int32_t* status) {
  if (blockIdx.x == 0) {
    plan_block(cu, row_ptr, pp, status, false);
    if (threadIdx.x == 0) *hdr = tag;  // flags 0: the forward kernel sets kAccZeroed
    return;
  }
  // the plan's per-position entries (block 0 has the tile ranges and lists):
  // qlo of every row, then kend of every row (fewer than 2^31 entries: the
  // plan's lists are at most kMaxListLen tiles)
  {
    const int total = __ldg(row_ptr + pp.B);
    const int nq = pp.B * pp.Lpad, ne = nq + pp.B * pp.Spad;
    for (int e = (blockIdx.x - 1) * blockDim.x + threadIdx.x; e < ne;
         e += (gridDim.x - 1) * blockDim.x) {
      const bool key = e >= nq;
      const int k = key ? e - nq : e;
      const int b = key ? k / pp.Spad : k / pp.Lpad;
      int n;
      const int32_t* c = row_list(cu, row_ptr, total, b, n);
      if (n < 1) n = 0;
      if (key)
        pp.kend[k] = kend_entry(c, n, k - b * pp.Spad);
      else
        pp.qlo[k] = qlo_entry(c, n, pp, k - b * pp.Lpad);
    }
  }
  for (long long i = (long long)(blockIdx.x - 1) * blockDim.x + threadIdx.x; i < n8;
       i += (long long)(gridDim.x - 1) * blockDim.x) {
    const uint4 x = v[i];
    v16[i] = make_uint4(bf16x2_to_f16x2(x.x), bf16x2_to_f16x2(x.y), bf16x2_to_f16x2(x.z),
                        bf16x2_to_f16x2(x.w));
  }
}

template <int D>
__global__ void __launch_bounds__(kPrepBwdThreads) prep_bwd_kernel(
    const int32_t* __restrict__ cu, const int32_t* __restrict__ row_ptr, const PlanPtrs pp,
    const WsTag* hdr, const WsTag expect, const __nv_bfloat16* __restrict__ out,
    const __half* __restrict__ out16, float o16_scale, const __nv_bfloat16* __restrict__ dout,
    const float* __restrict__ lse, int planes, int L, int Lq, float* __restrict__ nlse2o,
    float* __restrict__ ndeltao, float* __restrict__ dqacc, int32_t* status) {
  // the plan, the fp16 O and the zeroed accumulator the forward left
  // in the workspace belong to these inputs only if its header says so
  const bool same = same_tag(hdr, expect);
  if (blockIdx.x == 0) {
    if (!same) plan_block(cu, row_ptr, pp, status, true);
    return;
  }
  const bool zero = !(same && (hdr->flags & kAccZeroed) != 0);
  bwd_pre_rows<D>((long long)(blockIdx.x - 1) * blockDim.x + threadIdx.x, out,
                  same ? out16 : nullptr, o16_scale, dout, lse, planes, L, Lq, nlse2o, ndeltao,
                  zero ? dqacc : nullptr);
}

cudaError_t set_smem(const void* fn, size_t smem, int* done) {
  int dev = 0;
  cudaGetDevice(&dev);
  if (smem <= 48 * 1024 || dev >= 64 || done[dev]) return cudaSuccess;
  // the largest plan (kMaxListLen entries per list) needs 128 KB of keys,
  // its row bits and the boundary cache
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(sizeof(unsigned long long) * kMaxListLen +
                                                        512 * sizeof(uint32_t) +
                                                        kPlanCuCache * sizeof(int32_t)));
  if (e == cudaSuccess) done[dev] = 1;
  return e;
}

}  // namespace

cudaError_t launch_prep_fwd(const int32_t* cu, const int32_t* row_ptr, const PlanPtrs& pp,
                            const WsTag& tag, WsTag* hdr, const void* v, void* v16,
                            long long n_v, int32_t* status, int num_sms, cudaStream_t stream) {
  static int attr[64] = {};
  const size_t smem = plan_cta_smem(pp);
  cudaError_t e = set_smem(reinterpret_cast<const void*>(prep_fwd_kernel), smem, attr);
  if (e != cudaSuccess) return e;
  const long long n8 = n_v / 8;
  const long long want = (n8 + kPrepFwdThreads - 1) / kPrepFwdThreads;
  const int conv = static_cast<int>(want < 2LL * num_sms ? want : 2LL * num_sms);
  prep_fwd_kernel<<<1 + conv, kPrepFwdThreads, smem, stream>>>(
      cu, row_ptr, pp, tag, hdr, static_cast<const uint4*>(v), static_cast<uint4*>(v16), n8,
      status);
  return cudaGetLastError();
}

cudaError_t launch_prep_bwd(const BwdPrep& prep, const void* out, const void* out16,
                            float o16_scale, const void* dout, const float* lse, int D,
                            int planes, int L, int Lq, float* nlse2, float* ndelta, float* dqacc,
                            int32_t* status, cudaStream_t stream) {
  static int attr64[64] = {}, attr128[64] = {};
  const size_t smem = plan_cta_smem(prep.pp);
  const long long threads =
      (long long)planes * Lq * (D == 64 ? pre_threads_per_row<64>() : pre_threads_per_row<128>());
  const unsigned blocks =
      1 + static_cast<unsigned>((threads + kPrepBwdThreads - 1) / kPrepBwdThreads);
  const auto* o = static_cast<const __nv_bfloat16*>(out);
  const auto* ol = static_cast<const __half*>(out16);
  const auto* d = static_cast<const __nv_bfloat16*>(dout);
  cudaError_t e;
  if (D == 64) {
    e = set_smem(reinterpret_cast<const void*>(prep_bwd_kernel<64>), smem, attr64);
    if (e != cudaSuccess) return e;
    prep_bwd_kernel<64><<<blocks, kPrepBwdThreads, smem, stream>>>(
        prep.cu, prep.row_ptr, prep.pp, prep.hdr, prep.expect, o, ol, o16_scale, d, lse, planes,
        L, Lq, nlse2, ndelta, dqacc, status);
  } else {
    e = set_smem(reinterpret_cast<const void*>(prep_bwd_kernel<128>), smem, attr128);
    if (e != cudaSuccess) return e;
    prep_bwd_kernel<128><<<blocks, kPrepBwdThreads, smem, stream>>>(
        prep.cu, prep.row_ptr, prep.pp, prep.hdr, prep.expect, o, ol, o16_scale, d, lse, planes,
        L, Lq, nlse2, ndelta, dqacc, status);
  }
  return cudaGetLastError();
}

}  // namespace bd
