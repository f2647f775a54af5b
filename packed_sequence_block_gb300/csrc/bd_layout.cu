// Row-layout helpers around the attention path.
//
//  * doc_ids_from_seq_lens (page "nemo_automodel.components.models.glm5_next.cp"):
//    per-document lengths [B, documents], padded with padding_value, become
//    document ids [B, S]; padding entries take no number, the others are
//    numbered 1..n in order, positions past the last document get 0.
//  * document positions and validity (page
//    "nemo_automodel.components.models.inkling2.context_parallel",
//    unpack_row_layout): a document is a maximal run of equal non-zero ids;
//    its tokens get positions 0, 1, 2, ...; padding gets 0 and keep = 0.
//  * validate_document_positions (same page): among the kept tokens of a row,
//    the first may carry any position >= 0, a later one must carry 0, or its
//    predecessor's position + 1 when it directly follows it; after a gap it
//    must carry 0.
//  * the key/value rows the local queries [seq_start, seq_start + L) need
//    (page "nemo_automodel.components.distributed.blockdiag_cp", the
//    needed-only K/V exchange): [start of the segment of the first non-padding
//    local query, one past the last non-padding local query), and the part of
//    it inside each shard [r L, (r + 1) L) of the row.
#include <climits>

#include "bd_ptx.cuh"

namespace bd {

namespace {

constexpr int kLenThreads = 256;
constexpr int kScanThreads = 1024;
constexpr int kScanItems = 4;

// Exclusive scan of one value per thread over the block (sum, or max with
// identity LLONG_MIN); *total receives the block's reduction.  Every thread
// of the block must call it.
template <bool kMax>
__device__ __forceinline__ long long block_scan_excl(long long x, long long* warp_part,
                                                     long long* total) {
  const long long ident = kMax ? LLONG_MIN : 0;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  long long incl = x;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl = kMax ? (y > incl ? y : incl) : incl + y;
  }
  long long excl = __shfl_up_sync(0xffffffffu, incl, 1);
  if (lane == 0) excl = ident;
  if (lane == 31) warp_part[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    long long w = lane < nwarps ? warp_part[lane] : ident;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w = kMax ? (y > w ? y : w) : w + y;
    }
    if (lane < nwarps) warp_part[lane] = w;
  }
  __syncthreads();
  const long long wp = warp > 0 ? warp_part[warp - 1] : ident;
  *total = warp_part[nwarps - 1];
  excl = kMax ? (wp > excl ? wp : excl) : wp + excl;
  __syncthreads();  // warp_part is reused by the next call
  return excl;
}

}  // namespace

// Grid (ceil(S / 256), B).  Every block rebuilds its row's boundaries in shared
// memory from the lengths (short next to S), so an invalid row can be zeroed
// without a grid-wide sync.
__global__ void __launch_bounds__(kLenThreads) doc_ids_from_lens_kernel(
    const int32_t* __restrict__ lens_all, int ndocs, int S, int padding_value,
    int32_t* __restrict__ ids, int32_t* status) {
  extern __shared__ long long cu[];  // [ndocs + 1]: boundaries of the numbered documents
  __shared__ long long warp_part[32];
  const int b = blockIdx.y;
  const int32_t* lens = lens_all + (size_t)b * ndocs;
  if (threadIdx.x == 0) cu[0] = 0;
  int bad = 0;
  long long run = 0;  // total length of the documents of earlier chunks
  long long cnt = 0;  // documents of earlier chunks
  for (int j0 = 0; j0 < ndocs; j0 += kLenThreads) {
    const int j = j0 + threadIdx.x;
    long long len = 0, valid = 0;
    if (j < ndocs) {
      const int x = lens[j];
      if (x != padding_value) {
        valid = 1;
        if (x < 0) bad = 1; else len = x;
      }
    }
    long long tot_len, tot_cnt;
    const long long before_len = block_scan_excl<false>(len, warp_part, &tot_len);
    const long long before_cnt = block_scan_excl<false>(valid, warp_part, &tot_cnt);
    if (valid) cu[cnt + before_cnt + 1] = run + before_len + len;
    run += tot_len;
    cnt += tot_cnt;
  }
  bad = __syncthreads_or(bad || run > S);
  if (bad && blockIdx.x == 0 && threadIdx.x == 0) set_status(status, BD_ERR_INVALID_ARG);
  const int n = static_cast<int>(cnt);
  const int p = blockIdx.x * blockDim.x + threadIdx.x;
  if (p >= S) return;
  int32_t id = 0;
  if (!bad && cu[n] > p) {
    // first j in [1, n] with cu[j] > p: document j - 1, id j
    int lo = 1, hi = n;
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (cu[mid] > p) hi = mid; else lo = mid + 1;
    }
    id = lo;
  }
  ids[(size_t)b * S + p] = id;
}

constexpr int kChunk = kScanThreads * kScanItems;

// Largest q in [0, end) with pred(q), searched backwards one chunk at a time
// by the whole block; -1 when there is none.
template <typename Pred>
__device__ __forceinline__ long long last_before(int end, long long* warp_part, Pred pred) {
  for (int hi = end; hi > 0; hi -= kChunk) {
    const int lo = hi > kChunk ? hi - kChunk : 0;
    long long m = LLONG_MIN;
    for (int q = lo + threadIdx.x; q < hi; q += kScanThreads)
      if (pred(q)) m = q;
    long long tot;
    block_scan_excl<true>(m, warp_part, &tot);
    if (tot >= 0) return tot;
  }
  return -1;
}

// Grid (ceil(S / kChunk), B): one chunk of one row per block.  The start of
// the run holding p is the largest run start <= p: the chunk's own starts by
// a block scan, the run start in force at the chunk's first position by a
// backward search (position 0 always starts a run, so it ends).
__global__ void __launch_bounds__(kScanThreads) position_ids_kernel(
    const int32_t* __restrict__ ids_all, int S, int32_t* __restrict__ pos_all,
    uint8_t* __restrict__ keep_all) {
  __shared__ long long warp_part[32];
  const int b = blockIdx.y;
  const int32_t* ids = ids_all + (size_t)b * S;
  int32_t* pos = pos_all + (size_t)b * S;
  uint8_t* keep = keep_all + (size_t)b * S;
  const int c0 = blockIdx.x * kChunk;
  const long long carry =
      c0 == 0 ? 0 : last_before(c0, warp_part, [&](int q) { return q == 0 || ids[q] != ids[q - 1]; });
  const int p0 = c0 + threadIdx.x * kScanItems;
  int32_t id[kScanItems];
  long long st[kScanItems];
  long long m = LLONG_MIN;
#pragma unroll
  for (int u = 0; u < kScanItems; ++u) {
    const int p = p0 + u;
    id[u] = p < S ? ids[p] : 0;
    if (p < S && (p == 0 || id[u] != (u > 0 ? id[u - 1] : ids[p - 1]))) m = p;
    st[u] = m;
  }
  long long tot;
  long long before = block_scan_excl<true>(m, warp_part, &tot);
  if (carry > before) before = carry;
#pragma unroll
  for (int u = 0; u < kScanItems; ++u) {
    const int p = p0 + u;
    if (p < S) {
      const long long rs = st[u] > before ? st[u] : before;
      const bool k = id[u] != 0;
      pos[p] = k ? static_cast<int32_t>(p - rs) : 0;
      keep[p] = k ? 1 : 0;
    }
  }
}

// Grid (ceil(S / kChunk), B).  The previous kept column of p is the largest
// kept q < p: within the chunk by a block scan, before it by a backward
// search.  The smallest offending column of the row goes to bad[b] (bad must
// hold -1 or a column of the row; rows are reset by a preceding launch).
__global__ void __launch_bounds__(kScanThreads) validate_positions_kernel(
    const uint8_t* __restrict__ keep_all, const int32_t* __restrict__ pos_all, int S,
    int32_t* __restrict__ bad_all, int32_t* status) {
  __shared__ long long warp_part[32];
  __shared__ int first_bad;
  const int b = blockIdx.y;
  const uint8_t* keep = keep_all + (size_t)b * S;
  const int32_t* pos = pos_all + (size_t)b * S;
  if (threadIdx.x == 0) first_bad = INT_MAX;
  const int c0 = blockIdx.x * kChunk;
  const long long carry =
      c0 == 0 ? -1 : last_before(c0, warp_part, [&](int q) { return keep[q] != 0; });
  const int p0 = c0 + threadIdx.x * kScanItems;
  uint8_t k[kScanItems];
  long long m = LLONG_MIN;
#pragma unroll
  for (int u = 0; u < kScanItems; ++u) {
    const int p = p0 + u;
    k[u] = p < S ? keep[p] : 0;
    if (k[u]) m = p;
  }
  long long tot;
  long long prev = block_scan_excl<true>(m, warp_part, &tot);
  if (carry > prev) prev = carry;
#pragma unroll
  for (int u = 0; u < kScanItems; ++u) {
    const int p = p0 + u;
    if (p < S && k[u]) {
      const int32_t x = pos[p];
      bool ok;
      if (prev < 0) ok = x >= 0;
      else if (prev == p - 1) ok = x == 0 || x == pos[prev] + 1;
      else ok = x == 0;
      if (!ok) atomicMin(&first_bad, p);
      prev = p;
    }
  }
  __syncthreads();
  if (threadIdx.x == 0 && first_bad != INT_MAX) {
    atomicMin(reinterpret_cast<unsigned int*>(bad_all + b), static_cast<unsigned int>(first_bad));
    set_status(status, BD_ERR_INVALID_ARG);
  }
}

// first k in [0, n) with seg[k] <= x < seg[k + 1] (seg[0] = 0 <= x < seg[n])
__device__ __forceinline__ int segment_of(const int32_t* __restrict__ seg, int n, int x) {
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (seg[mid] <= x) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// One CTA per row: thread 0 finds [lo, hi); all threads fill the shard counts.
__global__ void __launch_bounds__(256) kv_range_kernel(
    const int32_t* __restrict__ seg_all, const int32_t* __restrict__ sid_all,
    const int32_t* __restrict__ nseg, int S, int L, int seq_start, int nshards,
    int32_t* __restrict__ range_all, int32_t* __restrict__ shard_all) {
  __shared__ int lo_s, hi_s;
  const int b = blockIdx.x;
  if (threadIdx.x == 0) {
    const int32_t* seg = seg_all + (size_t)b * (S + 1);
    const int32_t* sid = sid_all + (size_t)b * S;
    const int n = nseg[b];
    const int t0 = seq_start, t1 = seq_start + L;  // local queries [t0, t1)
    int lo = -1, hi = -1;
    // first non-padding segment that holds a local query, from the one holding t0;
    // between two document segments lies at most one padding segment
    for (int k = segment_of(seg, n, t0); k < n && seg[k] < t1; ++k) {
      if (sid[k] != 0) {
        lo = seg[k];
        break;
      }
    }
    for (int k = segment_of(seg, n, t1 - 1); k >= 0 && seg[k + 1] > t0; --k) {
      if (sid[k] != 0) {
        hi = min(seg[k + 1], t1);
        break;
      }
    }
    if (lo < 0) lo = hi = t0;
    lo_s = lo;
    hi_s = hi;
    range_all[2 * b] = lo;
    range_all[2 * b + 1] = hi;
  }
  __syncthreads();
  if (shard_all != nullptr) {
    const int lo = lo_s, hi = hi_s;
    for (int r = threadIdx.x; r < nshards; r += blockDim.x) {
      const long long a = max((long long)r * L, (long long)lo);
      const long long c = min(min((long long)(r + 1) * L, (long long)S), (long long)hi);
      shard_all[(size_t)b * nshards + r] = c > a ? static_cast<int32_t>(c - a) : 0;
    }
  }
}

cudaError_t launch_doc_ids_from_lens(const int32_t* lens, int B, int ndocs, int S,
                                     int padding_value, int32_t* ids, int32_t* status,
                                     cudaStream_t stream) {
  const size_t smem = sizeof(long long) * (static_cast<size_t>(ndocs) + 1);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(doc_ids_from_lens_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  dim3 grid(cdiv(S, kLenThreads), B);
  doc_ids_from_lens_kernel<<<grid, kLenThreads, smem, stream>>>(lens, ndocs, S, padding_value, ids,
                                                                status);
  return cudaGetLastError();
}

cudaError_t launch_position_ids(const int32_t* ids, int B, int S, int32_t* pos, uint8_t* keep,
                                cudaStream_t stream) {
  position_ids_kernel<<<dim3(cdiv(S, kChunk), B), kScanThreads, 0, stream>>>(ids, S, pos, keep);
  return cudaGetLastError();
}

cudaError_t launch_validate_positions(const uint8_t* keep, const int32_t* pos, int B, int S,
                                      int32_t* bad, int32_t* status, cudaStream_t stream) {
  // -1 (all bits set) is the largest unsigned value, so the blocks' unsigned
  // minimum leaves it only where no block found an offending column
  cudaError_t e = cudaMemsetAsync(bad, 0xff, sizeof(int32_t) * B, stream);
  if (e != cudaSuccess) return e;
  validate_positions_kernel<<<dim3(cdiv(S, kChunk), B), kScanThreads, 0, stream>>>(keep, pos, S,
                                                                                  bad, status);
  return cudaGetLastError();
}

cudaError_t launch_kv_range(const int32_t* seg, const int32_t* seg_ids, const int32_t* nseg,
                            int B, int S, int L, int seq_start, int32_t* range,
                            int32_t* shard_rows, cudaStream_t stream) {
  kv_range_kernel<<<B, 256, 0, stream>>>(seg, seg_ids, nseg, S, L, seq_start, cdiv(S, L), range,
                                         shard_rows);
  return cudaGetLastError();
}

}  // namespace bd
