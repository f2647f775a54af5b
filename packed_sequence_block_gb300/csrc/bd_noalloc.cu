// bd_attn_bwd_noalloc: the backward pass for callers that cannot allocate
// device memory.
//
// bd_attn_bwd_planned needs a caller-provided scratch buffer (the fp32 dq accumulator
// and per-row terms).  Some callers cannot provide one: code that runs inside
// a host runtime which reserves all device memory up front and forbids
// allocation afterwards (a cudaMalloc there can synchronise the device, stall
// other work, or fail once memory is fragmented).  This entry point uses a
// fixed scratch array that is part of the library image instead, so it
// allocates nothing; it launches the same kernels as bd_attn_bwd_planned.
#include <mutex>

#include "bd_internal.h"

namespace bd {
namespace {

// Scratch for problems whose backward workspace fits in BD_NOALLOC_SCRATCH_BYTES
// (16 MiB).  Every GPU that loads the library keeps this array for the life of
// the process.
constexpr size_t kNoAllocScratchBytes = BD_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_bwd_scratch[kNoAllocScratchBytes];

// Device address of g_bwd_scratch per device (the host-side symbol is only a
// stand-in and must never reach a kernel).  Looked up once per device, with
// that device current.
constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices] = {};
std::mutex g_scratch_mutex;

cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_bwd_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace bd

extern "C" {

int bd_attn_bwd_noalloc(const void* q, const void* k, const void* v, const void* out,
                        const void* out16, const float* lse, const void* dout, int B, int Hq,
                        int Hkv, int L, int S, int D, int seq_start, float scale, int enable_gqa,
                        void* plan, size_t plan_bytes, void* dq, void* dk, void* dv,
                        int32_t* dev_status, bd_stream_t stream) {
  if (B < 1 || Hq < 1 || L < 1 || D < 1) return BD_ERR_INVALID_ARG;
  const size_t need = bd_attn_bwd_planned_workspace_size(B, Hq, Hkv, L, S, D);
  if (need == 0) return BD_ERR_INVALID_ARG;
  if (need > bd::kNoAllocScratchBytes) return BD_ERR_WORKSPACE;
  // Arguments are checked by bd_attn_bwd_planned below before anything is launched;
  // the scratch address is looked up first only because it is an argument.
  void* scratch = nullptr;
  if (bd::scratch_address(&scratch) != cudaSuccess) return BD_ERR_CUDA;
  return bd_attn_bwd_planned(q, k, v, out, out16, lse, dout, B, Hq, Hkv, L, S, D, seq_start,
                             scale, enable_gqa, plan, plan_bytes, dq, dk, dv, scratch,
                             bd::kNoAllocScratchBytes, dev_status, stream);
}

}  // extern "C"
