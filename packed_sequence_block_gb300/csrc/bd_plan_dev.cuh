// Device helpers of the attention plan: binary searches over a row's
// boundaries, the ordering of the work lists, and the one-CTA plan
// builder that works straight from cumulative document boundaries.
//
// The mask is the per-document causal rule of cp_blockdiag_sdpa (page
// "nemo_automodel.components.distributed.blockdiag_cp"): the query at global
// position t attends keys j <= t of its own segment, and a query in a padding
// segment (id 0) attends nothing.  Ids from cumulative boundaries
// (doc_ids_from_cu_seqlens, page "nemo_automodel.components.models.glm5_next
// .cp") number the documents 1..n and give 0 past the last boundary, so the
// segments of such a row are its non-empty documents, then the padding run:
// the segment of position t < cu[n] is the document d with cu[d] <= t <
// cu[d + 1].  The builder below finds d by the same search that assigns the
// id and never stores the id array.
#pragma once

#include "bd_ptx.cuh"

namespace bd {

// first k with seg[k] > x, minus one: the segment holding x (seg[0] = 0 <= x < seg[n])
__device__ __forceinline__ int find_segment(const int32_t* __restrict__ seg, int n, int x) {
  int lo = 1, hi = n;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (seg[mid] > x) hi = mid; else lo = mid + 1;
  }
  return lo - 1;
}

// Key of entry i: cost descending, then index ascending (all keys distinct).
// The ranges may have been written earlier by the same block, so they are read
// through plain (coherent) loads.
__device__ __forceinline__ unsigned long long sort_key(const int32_t* range, int i) {
  const int cost = max(0, range[2 * i + 1] - range[2 * i] + 1);
  return (static_cast<unsigned long long>(0x7fffffffu - static_cast<unsigned>(cost)) << 32) |
         static_cast<unsigned>(i);
}

// Forward work lists whose every query block reaches at most this many key
// tiles keep the blocks in position order: each document's blocks then run
// side by side and share its K/V tiles in L2, and with units this short the
// longest-first order has little imbalance to remove (32-512-token documents:
// forward 450 us against 470; 1,024-token median documents: 138 us against
// 127 longest first).
constexpr int kShortFwdUnit = 8;

// Whether some entry of range[0..n) reaches more than kShortFwdUnit tiles.
// Every thread of the block calls it (it is a block-wide barrier).
__device__ __forceinline__ bool fwd_list_has_long_units(const int32_t* range, int n) {
  int any = 0;
  for (int i = threadIdx.x; i < n; i += blockDim.x)
    any |= range[2 * i + 1] - range[2 * i] + 1 > kShortFwdUnit;
  return __syncthreads_or(any) != 0;
}

// The forward list's key of entry i: longest first when `by_cost`, else the
// position order (the index).
__device__ __forceinline__ unsigned long long fwd_key(const int32_t* range, int i, bool by_cost) {
  return by_cost ? sort_key(range, i) : static_cast<unsigned long long>(i);
}

// Lists of up to kRankSortMax entries: the position of an entry is the number
// of smaller keys, one comparison pass per entry.
constexpr int kRankSortMax = 2048;

// order[0..n) = the entries by ascending key (keys unique, the entry's index
// in their low 32 bits).  Every thread of the block calls it.
__device__ inline void rank_order(const unsigned long long* keys, int n,
                                  int32_t* __restrict__ order) {
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    const unsigned long long ki = keys[i];
    int rank = 0;
    for (int j = 0; j < n; ++j) rank += keys[j] < ki;
    order[rank] = i;
  }
  __syncthreads();
}

// The same for longer lists: bitonic sort of keys[0..np) in place (np the next
// power of two >= n, entries past n hold ~0).
__device__ inline void bitonic_order(unsigned long long* keys, int n, int np,
                                     int32_t* __restrict__ order) {
  for (int size = 2; size <= np; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = threadIdx.x; i < np; i += blockDim.x) {
        const int j = i ^ stride;
        if (j > i) {
          const bool up = (i & size) == 0;
          const unsigned long long a = keys[i], c = keys[j];
          if ((a > c) == up) {
            keys[i] = c;
            keys[j] = a;
          }
        }
      }
      __syncthreads();
    }
  }
  for (int i = threadIdx.x; i < n; i += blockDim.x)
    order[i] = static_cast<int32_t>(keys[i] & 0xffffffffu);
  __syncthreads();
}

// A backward unit (key tile) opens a run unless it continues the previous
// tile's: same row, both non-empty, same last query tile.  The tiles of one
// document form one run (a tile shared by two documents joins the later one,
// whose last query tile it reaches).
__device__ __forceinline__ bool bwd_run_head(const int32_t* range, int i, int nkt) {
  const int lo = range[2 * i], hi = range[2 * i + 1];
  if (hi < lo || i % nkt == 0) return true;
  const int plo = range[2 * i - 2], phi = range[2 * i - 1];
  return phi < plo || phi != hi;
}

// Keys of the backward work list: documents by size, largest first (the size
// is the cost of the run's first, longest tile), each document's tiles
// together and longest first, empty tiles last; ties by index.  Units running
// side by side then share their Q/dO tiles and dq accumulator rows in L2
// (on a workload of 32-512-token documents the backward main kernel took
// 604 us in this order against 780 us longest-first).  The run heads come
// from a block-wide prefix maximum: each thread scans a contiguous chunk,
// then shuffles within warps and one pass over the warps' maxima (`scratch`:
// 64 ints of shared memory; blockDim.x a multiple of 32, at most 1024).
// Every thread of the block calls it.
__device__ inline void fill_bwd_keys(const int32_t* range, int n, int nkt,
                                     unsigned long long* keys, int32_t* scratch) {
  const int T = blockDim.x, t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int c = (n + T - 1) / T;
  const int b0 = min(n, t * c), b1 = min(n, b0 + c);
  int v = -1;  // the last run head in this thread's chunk
  for (int i = b0; i < b1; ++i)
    if (bwd_run_head(range, i, nkt)) v = i;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int u = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v = max(v, u);
  }
  if (lane == 31) scratch[warp] = v;
  __syncthreads();
  if (warp == 0) {
    int w = lane < (T >> 5) ? scratch[lane] : -1;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w = max(w, u);
    }
    scratch[32 + lane] = w;
  }
  __syncthreads();
  const int carry = warp > 0 ? scratch[32 + warp - 1] : -1;
  const int before = __shfl_up_sync(0xffffffffu, max(v, carry), 1);
  int head = lane > 0 ? before : carry;
  for (int i = b0; i < b1; ++i) {
    if (bwd_run_head(range, i, nkt)) head = i;
    const int lo = range[2 * i], hi = range[2 * i + 1];
    const int size = hi < lo ? 0 : min(range[2 * head + 1] - range[2 * head] + 1, 0xFFFFF);
    keys[i] = (static_cast<unsigned long long>(0xFFFFF - size) << 40) | static_cast<unsigned>(i);
  }
  __syncthreads();
}

// Order the forward work list into order[0..n): by cost (range length),
// longest first, ties by index, unless every entry is short (kShortFwdUnit:
// position order).  Every thread of the block calls it; `keys` holds the next
// power of two >= n entries of shared memory.
__device__ inline void sort_desc(const int32_t* range, int n, int32_t* __restrict__ order,
                                 unsigned long long* keys) {
  int np = 1;
  while (np < n) np <<= 1;
  const int m = n <= kRankSortMax ? n : np;
  const bool by_cost = fwd_list_has_long_units(range, n);
  for (int i = threadIdx.x; i < m; i += blockDim.x)
    keys[i] = i < n ? fwd_key(range, i, by_cost) : ~0ull;
  __syncthreads();
  if (n <= kRankSortMax)
    rank_order(keys, n, order);
  else
    bitonic_order(keys, n, np, order);
}

// The backward work list in the order of fill_bwd_keys.
__device__ inline void sort_bwd(const int32_t* range, int n, int nkt, int32_t* __restrict__ order,
                                unsigned long long* keys, int32_t* scratch) {
  int np = 1;
  while (np < n) np <<= 1;
  fill_bwd_keys(range, n, nkt, keys, scratch);
  if (n <= kRankSortMax) {
    rank_order(keys, n, order);
    return;
  }
  for (int i = n + threadIdx.x; i < np; i += blockDim.x) keys[i] = ~0ull;
  __syncthreads();
  bitonic_order(keys, n, np, order);
}

// Document index d of position x in a row with boundaries c[0..n] (valid, x < c[n]):
// the first j in [1, n] with c[j] > x, minus one.  `c` may point to shared or
// global memory.
__device__ __forceinline__ int find_doc(const int32_t* c, int n, int x) {
  int lo = 1, hi = n;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (c[mid] > x) hi = mid; else lo = mid + 1;
  }
  return lo - 1;
}

// Boundary entries the plan builder copies into shared memory (all rows
// together, then the row pointers); longer lists are read from global memory.
constexpr int kPlanCuCache = 4096;

// Row b's boundary list c[0..n] inside the array of `total` entries, or n = -1
// when the row pointers put it outside (the row then has no documents).
__device__ __forceinline__ const int32_t* row_list(const int32_t* cus, const int32_t* rps,
                                                   int total, int b, int& n) {
  const int base = rps[b];
  n = rps[b + 1] - base - 1;
  if (n < 0 || base < 0 || base + n + 1 > total) n = -1;
  return cus + (n >= 0 ? base : 0);
}

// The plan's per-position entries of a row with boundaries c[0..n] (n = 0:
// no documents): qlo of local query x, the start of its document (kPadLo for
// padding), and kend of key x, the end of its document (x itself for
// padding).  Searches stay inside c[0..n] whatever the list holds.
__device__ __forceinline__ int32_t qlo_entry(const int32_t* c, int n, const PlanPtrs& pp, int x) {
  const int last = n > 0 ? c[n] : 0;  // positions >= last are padding
  const int t = pp.seq_start + x;
  return (x < pp.L && t < last) ? c[find_doc(c, n, t)] : kPadLo;
}
__device__ __forceinline__ int32_t kend_entry(const int32_t* c, int n, int x) {
  const int last = n > 0 ? c[n] : 0;
  return x < last ? c[find_doc(c, n, x) + 1] : x;
}

// The whole plan of B rows in one CTA, from cumulative boundaries (rows as in
// bd_doc_ids_from_cu_seqlens: row b's list is cu[row_ptr[b] .. row_ptr[b+1]-1]).
// A row whose list does not start at 0, decreases, or ends past S is planned
// as all padding and BD_ERR_INVALID_ARG goes to *status, as its ids would be
// all 0.  Writes both tile ranges, both work-list orders, zeroes the work
// counters and, with write_rows, qlo and kend; without it other blocks write
// those with qlo_entry / kend_entry (a bad row's entries are then unspecified:
// its tiles are all empty, so no kernel reads them).  Every thread of the block
// calls it; `keys` is the sort's shared memory, `bad_rows` one bit per row
// (B <= 32 * bad_words), `cu_cache` kPlanCuCache entries of shared memory.
__device__ inline void build_plan_cta(const int32_t* __restrict__ cu,
                                      const int32_t* __restrict__ row_ptr, const PlanPtrs& pp,
                                      int32_t* status, unsigned long long* keys,
                                      uint32_t* bad_rows, int bad_words, int32_t* cu_cache,
                                      bool write_rows) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nwarps = blockDim.x >> 5;
  for (int i = threadIdx.x; i < bad_words; i += blockDim.x) bad_rows[i] = 0;
  if (threadIdx.x < 8) pp.sched[threadIdx.x] = 0;
  // Everything below reads the boundaries and row pointers from shared memory
  // when they fit (the blocks running beside this one stream through L1, so
  // global reads here would keep missing).
  const int total = __ldg(row_ptr + pp.B);
  const bool cached = total >= 0 && total + pp.B + 1 <= kPlanCuCache;
  if (cached) {
    for (int i = threadIdx.x; i < total; i += blockDim.x) cu_cache[i] = __ldg(cu + i);
    for (int i = threadIdx.x; i <= pp.B; i += blockDim.x) cu_cache[total + i] = __ldg(row_ptr + i);
  }
  const int32_t* cus = cached ? cu_cache : cu;
  const int32_t* rps = cached ? cu_cache + total : row_ptr;
  __syncthreads();
  // validity of each row's list, one warp per row
  for (int b = warp; b < pp.B; b += nwarps) {
    const int base = rps[b];
    const int n = rps[b + 1] - base - 1;
    // a row must also lie inside the boundary array row_ptr[B] declares
    int bad = n < 0 || base < 0 || base + n + 1 > total;
    for (int j = lane; !bad && j <= n; j += 32) {
      const int x = cus[base + j];
      if ((j == 0 && x != 0) || (j > 0 && x < cus[base + j - 1]) || x > pp.S) bad = 1;
    }
    if (__any_sync(0xffffffffu, bad) && lane == 0) {
      atomicOr(&bad_rows[b >> 5], 1u << (b & 31));
      set_status(status, BD_ERR_INVALID_ARG);
    }
  }
  __syncthreads();
  // Tile ranges, one thread per forward query block or backward key tile, from
  // the first and last positions of the tile that a document holds: document
  // starts and ends grow with the position, so the block's first valid query
  // has the smallest start and the tile's last valid key the largest end.
  const int nf = pp.B * pp.NQB, nb = pp.B * pp.NKT;
  for (int w = threadIdx.x; w < nf + nb; w += blockDim.x) {
    const bool fwd = w < nf;
    const int u = fwd ? w : w - nf;
    const int b = fwd ? u / pp.NQB : u / pp.NKT;
    const int blk = fwd ? u % pp.NQB : u % pp.NKT;
    const bool ok = ((bad_rows[b >> 5] >> (b & 31)) & 1u) == 0;
    int n;
    const int32_t* c = row_list(cus, rps, total, b, n);
    if (!ok || n < 1) n = 0;
    const int last = n > 0 ? c[n] : 0;  // positions >= last are padding
    if (fwd) {
      const int i0 = blk * pp.QROWS, t0 = pp.seq_start + i0;
      int lo = 0, hi = -1;
      if (i0 < pp.L && t0 < last) {
        lo = c[find_doc(c, n, t0)] / kBN;
        hi = min(pp.seq_start + min(pp.L, i0 + pp.QROWS) - 1, last - 1) / kBN;
      }
      pp.fwd_range[2 * u] = lo;
      pp.fwd_range[2 * u + 1] = hi;
    } else {
      const int p0 = blk * kBN;
      int a = 0, e = 0;
      if (p0 < last) {
        const int mx = c[find_doc(c, n, min(p0 + kBN, last) - 1) + 1];
        a = max(p0, pp.seq_start) - pp.seq_start;
        e = min(mx, pp.seq_start + pp.L) - pp.seq_start;
      }
      pp.bwd_range[2 * u] = (a < e) ? a / kBM : 0;
      pp.bwd_range[2 * u + 1] = (a < e) ? (e - 1) / kBM : -1;
    }
  }
  if (write_rows) {
    for (int b = 0; b < pp.B; ++b) {
      int n;
      const int32_t* c = row_list(cus, rps, total, b, n);
      if (((bad_rows[b >> 5] >> (b & 31)) & 1u) != 0 || n < 1) n = 0;
      for (int x = threadIdx.x; x < pp.Lpad; x += blockDim.x)
        pp.qlo[(size_t)b * pp.Lpad + x] = qlo_entry(c, n, pp, x);
      for (int x = threadIdx.x; x < pp.Spad; x += blockDim.x)
        pp.kend[(size_t)b * pp.Spad + x] = kend_entry(c, n, x);
    }
  }
  __threadfence_block();
  __syncthreads();
  // the boundary cache is free from here on: it holds the run-head scan
  if (nf <= kRankSortMax && nb <= kRankSortMax) {
    // both lists' keys side by side, then their ranks in one pass
    unsigned long long* kb = keys + nf;
    const bool by_cost = fwd_list_has_long_units(pp.fwd_range, nf);
    for (int i = threadIdx.x; i < nf; i += blockDim.x)
      keys[i] = fwd_key(pp.fwd_range, i, by_cost);
    fill_bwd_keys(pp.bwd_range, nb, pp.NKT, kb, cu_cache);
    for (int i = threadIdx.x; i < nf + nb; i += blockDim.x) {
      const bool f = i < nf;
      const unsigned long long* ks = f ? keys : kb;
      const int n = f ? nf : nb, idx = f ? i : i - nf;
      const unsigned long long ki = ks[idx];
      int rank = 0;
      for (int j = 0; j < n; ++j) rank += ks[j] < ki;
      (f ? pp.fwd_order : pp.bwd_order)[rank] = idx;
    }
    __syncthreads();
  } else {
    sort_desc(pp.fwd_range, nf, pp.fwd_order, keys);
    sort_bwd(pp.bwd_range, nb, pp.NKT, pp.bwd_order, keys, cu_cache);
  }
}

}  // namespace bd
