// Attention plan: mask bounds per row, non-empty tile ranges, ordered work
// lists (the forward's longest first, the backward's by document).
//
// The mask is the per-document causal rule of cp_blockdiag_sdpa (page
// "nemo_automodel.components.distributed.blockdiag_cp"): the query at global
// position t attends keys j <= t of its own segment, and a query in a padding
// segment (id 0) attends nothing.  Because segments are contiguous runs, each
// query row's key set is one interval [lo(t), t], and each key p is attended
// by the query interval [p, end of p's segment).  The kernels below turn the
// segment list into those bounds and into the tile ranges the attention
// kernels iterate over, so that fully masked tiles are never loaded.
#include "bd_plan_dev.cuh"

namespace bd {

// One warp per forward query block or backward key tile.  The warp of a
// query block first writes the mask bound qlo of each of its rows, the warp
// of a key tile the segment end kend of each of its keys (both from a binary
// search of the row's segment list), then reduces them to the block's
// non-empty tile range.  Warp 0 also zeroes the work counters.
__global__ void __launch_bounds__(256) plan_tiles_kernel(
    const int32_t* __restrict__ seg_all, const int32_t* __restrict__ seg_ids_all,
    const int32_t* __restrict__ nseg, int B, int L, int S, int seq_start, int NQB, int QROWS,
    int Lpad, int NKT, int Spad, int32_t* __restrict__ qlo, int32_t* __restrict__ kend,
    int32_t* __restrict__ fwd_range, int32_t* __restrict__ bwd_range,
    int32_t* __restrict__ sched) {
  const int w = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (w == 0 && lane < 8) sched[lane] = 0;
  const int nf = B * NQB;
  if (w < nf) {
    const int b = w / NQB, qb = w % NQB;
    const int32_t* seg = seg_all + (size_t)b * (S + 1);
    const int32_t* sid = seg_ids_all + (size_t)b * S;
    const int n = nseg[b];
    int mn = 0x7fffffff, mx = -1;
    for (int r = lane; r < QROWS; r += 32) {
      const int i = qb * QROWS + r;
      int32_t lo = kPadLo;
      if (i < L) {
        const int t = seq_start + i;
        const int k = find_segment(seg, n, t);
        if (sid[k] != 0) lo = seg[k];
      }
      qlo[(size_t)b * Lpad + i] = lo;
      if (lo != kPadLo) {
        mn = min(mn, lo);
        mx = max(mx, seq_start + i);
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      mn = min(mn, __shfl_xor_sync(0xffffffffu, mn, o));
      mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    }
    if (lane == 0) {
      const bool any = mx >= 0;
      fwd_range[2 * w] = any ? mn / kBN : 0;
      fwd_range[2 * w + 1] = any ? mx / kBN : -1;
    }
  } else if (w < nf + B * NKT) {
    const int u = w - nf;
    const int b = u / NKT, kt = u % NKT;
    const int32_t* seg = seg_all + (size_t)b * (S + 1);
    const int32_t* sid = seg_ids_all + (size_t)b * S;
    const int n = nseg[b];
    int mn = 0x7fffffff, mx = -1;
    for (int r = lane; r < kBN; r += 32) {
      const int p = kt * kBN + r;
      int32_t e = p;
      if (p < S) {
        const int k = find_segment(seg, n, p);
        if (sid[k] != 0) e = seg[k + 1];
      }
      kend[(size_t)b * Spad + p] = e;
      if (e > p) {
        mn = min(mn, p);
        mx = max(mx, e);
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      mn = min(mn, __shfl_xor_sync(0xffffffffu, mn, o));
      mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    }
    if (lane == 0) {
      int a = 0, c = 0;
      if (mx >= 0) {
        a = max(mn, seq_start) - seq_start;
        c = min(mx, seq_start + L) - seq_start;
      }
      bwd_range[2 * u] = (a < c) ? a / kBM : 0;
      bwd_range[2 * u + 1] = (a < c) ? (c - 1) / kBM : -1;
    }
  }
}

// Sort the forward work list by cost (range length), longest first, and the
// backward one by document (fill_bwd_keys); ties by index.  One CTA; 64-bit
// keys in shared memory, then the run-head scan's ints.
constexpr int kSortThreads = 1024;

__global__ void __launch_bounds__(kSortThreads) plan_sort_kernel(const int32_t* fwd_range, int nf,
                                                                 int32_t* fwd_order,
                                                                 const int32_t* bwd_range, int nb,
                                                                 int nkt, int32_t* bwd_order,
                                                                 int np) {
  extern __shared__ unsigned long long keys[];
  int32_t* scratch = reinterpret_cast<int32_t*>(keys + np);
  sort_desc(fwd_range, nf, fwd_order, keys);
  sort_bwd(bwd_range, nb, nkt, bwd_order, keys, scratch);
}

PlanPtrs plan_ptrs(void* plan, int B, int Hq, int Hkv, int L, int S, int seq_start) {
  const PlanLayout pl = plan_layout(B, Hq, Hkv, L, S);
  char* base = static_cast<char*>(plan);
  PlanPtrs pp{};
  pp.B = B;
  pp.L = L;
  pp.S = S;
  pp.seq_start = seq_start;
  pp.NQB = pl.NQB;
  pp.QROWS = pl.QROWS;
  pp.Lpad = pl.Lpad;
  pp.NKT = pl.NKT;
  pp.Spad = pl.Spad;
  pp.qlo = reinterpret_cast<int32_t*>(base + pl.qlo);
  pp.kend = reinterpret_cast<int32_t*>(base + pl.kend);
  pp.fwd_range = reinterpret_cast<int32_t*>(base + pl.fwd_range);
  pp.bwd_range = reinterpret_cast<int32_t*>(base + pl.bwd_range);
  pp.fwd_order = reinterpret_cast<int32_t*>(base + pl.fwd_order);
  pp.bwd_order = reinterpret_cast<int32_t*>(base + pl.bwd_order);
  pp.sched = reinterpret_cast<int32_t*>(base + pl.sched);
  return pp;
}

size_t plan_cta_smem(const PlanPtrs& pp) {
  const int nf = pp.B * pp.NQB, nb = pp.B * pp.NKT;
  int np = 1;
  while (np < max(nf, nb)) np <<= 1;
  // the keys of both lists side by side (rank sort), or one list padded to a
  // power of two (bitonic sort)
  const int nkeys = (nf <= kRankSortMax && nb <= kRankSortMax) ? max(np, nf + nb) : np;
  return sizeof(unsigned long long) * nkeys + sizeof(uint32_t) * ((pp.B + 31) / 32) +
         sizeof(int32_t) * kPlanCuCache;
}

cudaError_t launch_plan(const int32_t* seg, const int32_t* seg_ids, const int32_t* nseg, int B,
                        int Hq, int Hkv, int L, int S, int seq_start, void* plan,
                        cudaStream_t stream) {
  const PlanLayout pl = plan_layout(B, Hq, Hkv, L, S);
  char* base = static_cast<char*>(plan);
  int32_t* qlo = reinterpret_cast<int32_t*>(base + pl.qlo);
  int32_t* kend = reinterpret_cast<int32_t*>(base + pl.kend);
  int32_t* fr = reinterpret_cast<int32_t*>(base + pl.fwd_range);
  int32_t* br = reinterpret_cast<int32_t*>(base + pl.bwd_range);
  int32_t* fo = reinterpret_cast<int32_t*>(base + pl.fwd_order);
  int32_t* bo = reinterpret_cast<int32_t*>(base + pl.bwd_order);
  int32_t* sc = reinterpret_cast<int32_t*>(base + pl.sched);

  const int warps = B * pl.NQB + B * pl.NKT;
  plan_tiles_kernel<<<cdiv(warps * 32, 256), 256, 0, stream>>>(
      seg, seg_ids, nseg, B, L, S, seq_start, pl.NQB, pl.QROWS, pl.Lpad, pl.NKT, pl.Spad, qlo,
      kend, fr, br, sc);
  const int nf = B * pl.NQB, nb = B * pl.NKT;
  int np = 1;
  while (np < max(nf, nb)) np <<= 1;
  const size_t smem = sizeof(unsigned long long) * np + sizeof(int32_t) * kSortThreads;
  static bool attr_set[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (smem > 48 * 1024 && dev < 64 && !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(
        plan_sort_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
        static_cast<int>(sizeof(unsigned long long) * kMaxListLen + sizeof(int32_t) * kSortThreads));
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  plan_sort_kernel<<<1, kSortThreads, smem, stream>>>(fr, nf, fo, br, nb, pl.NKT, bo, np);
  return cudaGetLastError();
}

}  // namespace bd
