// Internal declarations shared by the library's translation units: constants,
// the plan buffer layout and the kernel launchers called by the C ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/bd_attn.h"

namespace bd {

// Tile sizes: 128 query rows x 128 keys per MMA tile.
constexpr int kBM = 128;
constexpr int kBN = 128;

// Device-side waits give up after this long (a healthy wait lasts microseconds).
constexpr unsigned long long kWaitTimeoutNs = 2000000000ull;

// Mask lower bound of a query row that attends nothing (padding / past L).
constexpr int32_t kPadLo = 0x7fffffff;

// Largest work list the single-CTA sorter handles.
constexpr int kMaxListLen = 16384;

inline size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }
inline int cdiv(int a, int b) { return (a + b - 1) / b; }

// Plan buffer layout (byte offsets from the plan base, each 256-aligned).
//   qlo       int32 [B, Lpad]  segment start of query row i (global position),
//                              kPadLo when the row attends nothing
//   kend      int32 [B, Spad]  end of the segment holding key p, or p itself
//                              for a padding key (no query attends it)
//   fwd_range int32 [B*NQB, 2] non-empty key-tile range [lo, hi] of each
//                              query block (hi < lo when empty)
//   bwd_range int32 [B*NKT, 2] query-tile range [lo, hi] of each key tile
//   fwd_order int32 [B*NQB]    query blocks sorted by cost, longest first
//   bwd_order int32 [B*NKT]    key tiles sorted by cost, longest first
//   sched     int32 [8]        work counters: [0..1] forward, [2..3] backward
//                              (next unit, finished CTAs); zeroed by the
//                              planner, reset by the last CTA of each launch
// A forward query block is 128 rows when Hq/Hkv is even (its two halves are
// two heads of one group) and 256 rows when it is odd (two consecutive
// 128-row tiles of one head).
struct PlanLayout {
  int NQB, NKT, QROWS, Lpad, Spad;
  size_t qlo, kend, fwd_range, bwd_range, fwd_order, bwd_order, sched, total;
};

inline PlanLayout plan_layout(int B, int Hq, int Hkv, int L, int S) {
  PlanLayout p{};
  const int G = Hkv > 0 ? Hq / Hkv : 1;
  p.QROWS = (G % 2 == 0) ? kBM : 2 * kBM;
  p.NQB = cdiv(L, p.QROWS);
  p.NKT = cdiv(S, kBN);
  p.Lpad = p.NQB * p.QROWS;
  p.Spad = p.NKT * kBN;
  size_t off = 0;
  p.qlo = off;       off = align256(off + sizeof(int32_t) * (size_t)B * p.Lpad);
  p.kend = off;      off = align256(off + sizeof(int32_t) * (size_t)B * p.Spad);
  p.fwd_range = off; off = align256(off + sizeof(int32_t) * 2 * (size_t)B * p.NQB);
  p.bwd_range = off; off = align256(off + sizeof(int32_t) * 2 * (size_t)B * p.NKT);
  p.fwd_order = off; off = align256(off + sizeof(int32_t) * (size_t)B * p.NQB);
  p.bwd_order = off; off = align256(off + sizeof(int32_t) * (size_t)B * p.NKT);
  p.sched = off;     off = align256(off + sizeof(int32_t) * 8);
  p.total = off;
  return p;
}

// Backward workspace: fp32 dq accumulator [B,Hq,L,D], then per-row
// -lse * log2 e [B,Hq,Lq] followed by -Delta [B,Hq,Lq] (Lq = ceil(L/128)*128).
struct BwdLayout {
  int Lq;
  size_t dqacc, lsed, total;
};

inline BwdLayout bwd_layout(int B, int Hq, int Hkv, int L, int S, int D) {
  BwdLayout w{};
  w.Lq = cdiv(L, kBM) * kBM;
  size_t off = 0;
  w.dqacc = off; off = align256(off + sizeof(float) * (size_t)B * Hq * L * D);
  w.lsed = off;  off = align256(off + sizeof(float) * 2 * (size_t)B * Hq * w.Lq);
  w.total = off;
  return w;
}

// Attention dropout: element (plane, query position t, key position j) is kept
// iff the 16-bit half j & 1 of word (j & 7) >> 1 of Philox4x32-10(counter
// (j >> 3, t, plane, offset), key (k0, k1)) is >= threshold = floor(p * 2^16);
// kept weights are scaled by rp = 1 / (1 - threshold / 2^16).
// rk holds the key schedule, round r's key words at rk[2r], rk[2r + 1]
// (k0 + r 0x9E3779B9, k1 + r 0xBB67AE85), read by the kernels from their
// parameter space.
struct DropoutArgs {
  bool on = false;
  uint32_t threshold = 0;
  float rp = 1.f;  // 1 / (1 - p)
  uint32_t offset = 0;
  uint32_t rk[20] = {};
};

struct AttnDims {
  int B, Hq, Hkv, L, S, D, seq_start;
  float scale;        // softmax scale (resolved, > 0)
  float scale_log2;   // scale * log2(e)
  DropoutArgs drop;
};

// ---- launchers (each enqueues on `stream`; returns the launch error) ----

cudaError_t launch_doc_ids(const int32_t* cu, const int32_t* row_ptr, int B, int S, int32_t* ids,
                           int32_t* status, cudaStream_t stream);
cudaError_t launch_segments(const int32_t* ids, int B, int S, int32_t* seg, int32_t* seg_ids,
                            int32_t* nseg, cudaStream_t stream);
cudaError_t launch_doc_ids_from_lens(const int32_t* lens, int B, int ndocs, int S,
                                     int padding_value, int32_t* ids, int32_t* status,
                                     cudaStream_t stream);
cudaError_t launch_position_ids(const int32_t* ids, int B, int S, int32_t* pos, uint8_t* keep,
                                cudaStream_t stream);
cudaError_t launch_validate_positions(const uint8_t* keep, const int32_t* pos, int B, int S,
                                      int32_t* bad, int32_t* status, cudaStream_t stream);
cudaError_t launch_kv_range(const int32_t* seg, const int32_t* seg_ids, const int32_t* nseg,
                            int B, int S, int L, int seq_start, int32_t* range,
                            int32_t* shard_rows, cudaStream_t stream);
// Largest documents dimension bd_doc_ids_from_seq_lens accepts.
constexpr int kMaxDocsPerRow = 8192;
cudaError_t launch_plan(const int32_t* seg, const int32_t* seg_ids, const int32_t* nseg, int B,
                        int Hq, int Hkv, int L, int S, int seq_start, void* plan,
                        cudaStream_t stream);

// Tensor maps for q/k/v-like tensors [planes, rows, D] (bf16, 128-byte swizzle,
// box 64 x 128 x 1).  Returns false when the driver rejects the map.
bool make_tmap_bf16(CUtensorMap* map, const void* base, int planes, int rows, int D);
// bf16 [planes, rows, D] written by TMA stores of 32 x 32 boxes (64-byte swizzle).
bool make_tmap_out(CUtensorMap* map, const void* base, int planes, int rows, int D);
// The same for fp16 data.
bool make_tmap_f16(CUtensorMap* map, const void* base, int planes, int rows, int D);
// Tensor map for the fp32 dq accumulator [planes, rows, D] (128-byte swizzle,
// box 32 x 128 x 1), the target of the backward's TMA reduce-adds.
bool make_tmap_dqacc(CUtensorMap* map, void* base, int planes, int rows, int D);

// Converts v to fp16 into v16 (the map tv describes v16), then runs the forward.
cudaError_t launch_fwd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const CUtensorMap& to, const CUtensorMap& tol,
                       const AttnDims& d, void* plan, const void* v, void* v16, void* out,
                       void* out_lo, float* lse, int32_t* status, int num_sms,
                       cudaStream_t stream);
// Backward stages (bit mask): per-row terms + accumulator zeroing, the main
// dK/dV/dQ kernel, and the dq conversion.
constexpr int kBwdPrepare = 1, kBwdMain = 2, kBwdFinish = 4;

cudaError_t launch_bwd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const CUtensorMap& tdo, const CUtensorMap& tdq, const AttnDims& d,
                       void* plan, const void* out, const void* out_lo, const float* lse,
                       const void* dout, void* dq, void* dk,
                       void* dv, void* workspace, int32_t* status, int stages, int num_sms,
                       cudaStream_t stream);

}  // namespace bd
