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

static_assert(kWaitTimeoutNs < (1ull << 32), "the wait limit travels as 32 bits");

// Test hook for the bounded waits (bd_test_arm_wait_timeout): the next launch
// of the chosen kernel from this host thread withholds its producer's first
// arrival and uses a shorter wait limit.  take_wait_test() returns the
// launch's limit in nanoseconds and whether to withhold, and disarms.
constexpr int kWaitTestFwd = 1, kWaitTestBwd = 2;
void arm_wait_test(int which, uint32_t limit_ns);
uint32_t take_wait_test(int which, int* withhold);

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
//   bwd_order int32 [B*NKT]    key tiles by document: largest documents first, each
//                              document's tiles together, longest first
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

// Workspace of the single-call entry points (bd_attn_fwd / bd_attn_bwd, which
// take cumulative boundaries): a 256-byte header, the plan, the fp16 copy of
// v, the forward's fp16 copy of O (out16), then the backward workspace.
// Every part starts on a 256-byte boundary.
struct WsLayout {
  PlanLayout plan;
  BwdLayout bwd;
  size_t hdr, plan_off, v16, out16, bwd_off, total;
};

inline WsLayout ws_layout(int B, int Hq, int Hkv, int L, int S, int D) {
  WsLayout w{};
  w.plan = plan_layout(B, Hq, Hkv, L, S);
  w.bwd = bwd_layout(B, Hq, Hkv, L, S, D);
  size_t off = 0;
  w.hdr = off;      off = 256;
  w.plan_off = off; off = align256(off + w.plan.total);
  w.v16 = off;      off = align256(off + 2 * (size_t)B * Hkv * S * D);
  w.out16 = off;   off = align256(off + 2 * (size_t)B * Hq * L * D);
  w.bwd_off = off;  off = align256(off + w.bwd.total);
  w.total = off;
  return w;
}

// What the single-call forward records in the workspace header: the shapes,
// the boundaries it planned from and the output it wrote.  The backward
// reuses the plan and the fp16 O kept in the workspace only when the
// header names the same shapes, boundaries, out and lse; otherwise it
// rebuilds the plan and forms Delta from the bf16 output alone.  `flags`
// (not part of the match) has kAccZeroed set by the forward kernel once it
// has zeroed the backward's dq accumulator, and cleared by the backward main
// kernel, which leaves the accumulator holding sums.
struct WsTag {
  uint32_t magic;
  int32_t B, Hq, Hkv, L, S, D, seq_start;
  unsigned long long out, lse, cu, row_ptr;
  uint32_t flags;
};
constexpr uint32_t kWsMagic = 0x42445733u;  // "BDW3"
constexpr uint32_t kAccZeroed = 1u;

// Where the plan builder writes (device pointers into a plan buffer).
struct PlanPtrs {
  int B, L, S, seq_start, NQB, QROWS, Lpad, NKT, Spad;
  int32_t *qlo, *kend, *fwd_range, *bwd_range, *fwd_order, *bwd_order, *sched;
};
PlanPtrs plan_ptrs(void* plan, int B, int Hq, int Hkv, int L, int S, int seq_start);
// Dynamic shared memory the one-CTA plan builder needs (sorting keys).
size_t plan_cta_smem(const PlanPtrs& pp);

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
// 16-bit [planes, rows, D] (out: bf16, out16: fp16) written by TMA stores of
// 32 x 32 boxes (64-byte swizzle).
bool make_tmap_out(CUtensorMap* map, const void* base, int planes, int rows, int D,
                   CUtensorMapDataType type);
// The same for fp16 data.
bool make_tmap_f16(CUtensorMap* map, const void* base, int planes, int rows, int D);
// Tensor map for the fp32 dq accumulator [planes, rows, D] (128-byte swizzle,
// box 32 x 128 x 1), the target of the backward's TMA reduce-adds.
bool make_tmap_dqacc(CUtensorMap* map, void* base, int planes, int rows, int D);

// v (bf16) -> v16 (fp16), the P V operand of the forward.
cudaError_t launch_v_to_f16(const void* v, void* v16, long long n, int num_sms,
                            cudaStream_t stream);
// The forward kernel alone (v16 already written; the map tv describes it).
// `acc`, when not NULL, is a buffer of acc_bytes (a multiple of 16) that the
// kernel's otherwise idle warps zero while it runs; `acc_flags` (or NULL)
// then gets kAccZeroed once every CTA finished without an error.
cudaError_t launch_fwd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const CUtensorMap& to, const CUtensorMap& to16,
                       const AttnDims& d, void* plan, void* out,
                       void* out16, float* lse, int32_t* status, int num_sms,
                       cudaStream_t stream, void* acc = nullptr, size_t acc_bytes = 0,
                       uint32_t* acc_flags = nullptr);
// One launch before the single-call forward: block 0 builds the plan from the
// cumulative boundaries (validating them) and writes the workspace tag; the
// other blocks convert v to fp16.
cudaError_t launch_prep_fwd(const int32_t* cu, const int32_t* row_ptr, const PlanPtrs& pp,
                            const WsTag& tag, WsTag* hdr, const void* v, void* v16,
                            long long n_v, int32_t* status, int num_sms, cudaStream_t stream);
// Backward stages (bit mask): per-row terms + accumulator zeroing, the main
// dK/dV/dQ kernel, and the dq conversion.
constexpr int kBwdPrepare = 1, kBwdMain = 2, kBwdFinish = 4;

// For the single-call backward: stage 1 also builds the plan from the
// cumulative boundaries (block 0 of the same launch), and takes the fp16 O
// from the workspace only when the header carries `expect`.
struct BwdPrep {
  const int32_t* cu;
  const int32_t* row_ptr;
  PlanPtrs pp;
  WsTag* hdr;
  WsTag expect;
};

cudaError_t launch_bwd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const CUtensorMap& tdo, const CUtensorMap& tdq, const AttnDims& d,
                       void* plan, const void* out, const void* out16, const float* lse,
                       const void* dout, void* dq, void* dk,
                       void* dv, void* workspace, int32_t* status, int stages, int num_sms,
                       cudaStream_t stream, const BwdPrep* prep = nullptr);

// Stage 1 of the single-call backward (one launch): block 0 builds the plan
// unless the workspace header shows the forward's plan for the same inputs;
// the other blocks write -lse log2 e and -Delta per row and zero the dq
// accumulator unless the header says the forward already did (the rows'
// terms as bwd_pre_kernel writes them).
cudaError_t launch_prep_bwd(const BwdPrep& prep, const void* out, const void* out16,
                            float o16_scale, const void* dout, const float* lse, int D,
                            int planes, int L, int Lq, float* nlse2, float* ndelta, float* dqacc,
                            int32_t* status, cudaStream_t stream);

}  // namespace bd
