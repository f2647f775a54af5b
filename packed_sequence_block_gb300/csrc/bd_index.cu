// Document ids from cumulative boundaries and segment boundaries from ids.
//
// doc_ids_from_cu_seqlens / segment_cu_seqlens / _PAD_DOC_ID = 0 on the page
// "nemo_automodel.components.models.glm5_next.cp": position p of a row gets
// d + 1 when cu[d] <= p < cu[d+1] and 0 past the last boundary; segments are
// the maximal runs of equal ids covering the whole row.
#include "bd_ptx.cuh"

namespace bd {

// One block of 256 positions of one row.  Every block re-checks its row's
// boundary list (cheap: the list is short next to S) so that an invalid row
// can be zeroed without a grid-wide sync.
__global__ void __launch_bounds__(256) doc_ids_kernel(const int32_t* __restrict__ cu,
                                                      const int32_t* __restrict__ row_ptr,
                                                      int S, int32_t* __restrict__ ids,
                                                      int32_t* status) {
  const int b = blockIdx.y;
  const int base = row_ptr[b];
  const int n = row_ptr[b + 1] - base - 1;  // number of documents
  const int32_t* c = cu + base;
  int bad = (n < 0) ? 1 : 0;
  if (!bad) {
    for (int j = threadIdx.x; j <= n; j += blockDim.x) {
      const int x = c[j];
      if ((j == 0 && x != 0) || (j > 0 && x < c[j - 1]) || x > S) bad = 1;
    }
  }
  bad = __syncthreads_or(bad);
  if (bad && blockIdx.x == 0 && threadIdx.x == 0) set_status(status, BD_ERR_INVALID_ARG);

  const int p = blockIdx.x * blockDim.x + threadIdx.x;
  if (p >= S) return;
  int32_t id = 0;
  if (!bad && c[n] > p) {
    // first j in [1, n] with c[j] > p; the document is j - 1, its id j
    int lo = 1, hi = n;
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (c[mid] > p) hi = mid; else lo = mid + 1;
    }
    id = lo;
  }
  ids[(size_t)b * S + p] = id;
}

// One CTA per row: flag run starts, block-wide scan, scatter.
constexpr int kSegThreads = 1024;
constexpr int kSegItems = 4;

__global__ void __launch_bounds__(kSegThreads) segments_kernel(const int32_t* __restrict__ ids_all,
                                                               int S, int32_t* __restrict__ seg_all,
                                                               int32_t* __restrict__ seg_ids_all,
                                                               int32_t* __restrict__ nseg) {
  __shared__ int warp_sums[kSegThreads / 32];
  __shared__ int carry;
  const int b = blockIdx.x;
  const int32_t* ids = ids_all + (size_t)b * S;
  int32_t* seg = seg_all + (size_t)b * (S + 1);
  int32_t* seg_ids = seg_ids_all + (size_t)b * S;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) carry = 0;
  __syncthreads();
  for (int chunk = 0; chunk < S; chunk += kSegThreads * kSegItems) {
    const int p0 = chunk + threadIdx.x * kSegItems;
    int flags[kSegItems];
    int cnt = 0;
#pragma unroll
    for (int u = 0; u < kSegItems; ++u) {
      const int p = p0 + u;
      flags[u] = (p < S) && (p == 0 || ids[p] != ids[p - 1]);
      cnt += flags[u];
    }
    // inclusive warp scan of cnt
    int x = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) warp_sums[warp] = x;
    __syncthreads();
    if (warp == 0) {
      int w = warp_sums[lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, w, o);
        if (lane >= o) w += y;
      }
      warp_sums[lane] = w;  // inclusive over warps
    }
    __syncthreads();
    int rank = carry + (warp > 0 ? warp_sums[warp - 1] : 0) + x - cnt;
#pragma unroll
    for (int u = 0; u < kSegItems; ++u) {
      if (flags[u]) {
        const int p = p0 + u;
        seg[rank] = p;
        seg_ids[rank] = ids[p];
        ++rank;
      }
    }
    __syncthreads();
    if (threadIdx.x == 0) carry += warp_sums[31];
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    seg[carry] = S;
    nseg[b] = carry;
  }
}

cudaError_t launch_doc_ids(const int32_t* cu, const int32_t* row_ptr, int B, int S, int32_t* ids,
                           int32_t* status, cudaStream_t stream) {
  dim3 grid(cdiv(S, 256), B);
  doc_ids_kernel<<<grid, 256, 0, stream>>>(cu, row_ptr, S, ids, status);
  return cudaGetLastError();
}

cudaError_t launch_segments(const int32_t* ids, int B, int S, int32_t* seg, int32_t* seg_ids,
                            int32_t* nseg, cudaStream_t stream) {
  segments_kernel<<<B, kSegThreads, 0, stream>>>(ids, S, seg, seg_ids, nseg);
  return cudaGetLastError();
}

}  // namespace bd
