// The library's C ABI (declared in include/bd_attn.h): argument checks,
// TMA tensor maps and launches.  No call allocates, frees or synchronises
// except bd_get_device_status, which exists to read the status word back.
#include <cudaTypedefs.h>

#include <cmath>
#include <mutex>

#include "bd_internal.h"

namespace bd {

namespace {

PFN_cuTensorMapEncodeTiled_v12000 tmap_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

int num_sms_current() {
  static int cache[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < 64 && cache[dev] > 0) return cache[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < 64) cache[dev] = n;
  return n;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Shapes shared by the attention entry points.
int check_dims(int B, int Hq, int Hkv, int L, int S, int D, int seq_start, int enable_gqa) {
  if (B < 1 || Hq < 1 || Hkv < 1 || L < 1 || S < 1 || D < 1 || seq_start < 0)
    return BD_ERR_INVALID_ARG;
  if (static_cast<long long>(seq_start) + L > S) return BD_ERR_INVALID_ARG;
  if (Hq % Hkv != 0) return BD_ERR_INVALID_ARG;
  if (Hq != Hkv && !enable_gqa) return BD_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return BD_ERR_UNSUPPORTED;
  // TMA planes/rows and the int offsets used on the device
  if (static_cast<long long>(B) * Hq * L * D >= (1ll << 40)) return BD_ERR_UNSUPPORTED;
  if (static_cast<long long>(B) * Hq > (1ll << 30) || S > (1 << 30)) return BD_ERR_UNSUPPORTED;
  return BD_OK;
}

int check_plan_lists(int B, int Hq, int Hkv, int L, int S) {
  const PlanLayout pl = plan_layout(B, Hq, Hkv, L, S);
  if (static_cast<long long>(B) * pl.NQB > kMaxListLen ||
      static_cast<long long>(B) * pl.NKT > kMaxListLen)
    return BD_ERR_UNSUPPORTED;
  return BD_OK;
}

AttnDims resolve(int B, int Hq, int Hkv, int L, int S, int D, int seq_start, float scale) {
  AttnDims d{B, Hq, Hkv, L, S, D, seq_start, scale, 0.f, DropoutArgs{}};
  if (!(scale > 0.f) || !std::isfinite(scale)) d.scale = 1.0f / std::sqrt(static_cast<float>(D));
  d.scale_log2 = d.scale * 1.4426950408889634f;
  return d;
}

// Dropout arguments: p in [0, 1); an element is kept iff its 16-bit Philox
// value is >= floor(p * 2^16), so the drop probability is p' = that
// threshold / 2^16 and kept weights are scaled by 1 / (1 - p').  A p below
// 2^-16 drops nothing and runs the kernels without dropout.
int make_dropout(double p, uint64_t seed, uint32_t offset, DropoutArgs* out) {
  if (!(p >= 0.0 && p < 1.0)) return BD_ERR_INVALID_ARG;
  DropoutArgs d;
  const double thr = std::floor(p * 65536.0);
  d.threshold = thr >= 65535.0 ? 65535u : static_cast<uint32_t>(thr);
  d.on = d.threshold > 0;
  d.rp = static_cast<float>(1.0 / (1.0 - d.threshold / 65536.0));
  uint32_t k0 = static_cast<uint32_t>(seed & 0xffffffffu);
  uint32_t k1 = static_cast<uint32_t>(seed >> 32);
  for (int r = 0; r < 10; ++r) {  // the Philox key schedule
    d.rk[2 * r] = k0;
    d.rk[2 * r + 1] = k1;
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  d.offset = offset;
  *out = d;
  return BD_OK;
}


}  // namespace

static bool make_tmap_16bit(CUtensorMap* map, const void* base, int planes, int rows, int D,
                            CUtensorMapDataType dtype) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tmap_encoder();
  if (enc == nullptr) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(rows),
                        static_cast<cuuint64_t>(planes)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2,
                           static_cast<cuuint64_t>(rows) * D * 2};
  cuuint32_t box[3] = {64, 128, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, dtype, 3, const_cast<void*>(base), dims,
                   strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

namespace {
// One-shot wait-test requests of this host thread, per kernel (index 1: forward,
// 2: backward main); 0 means none.
thread_local uint32_t t_wait_test_ns[3] = {0, 0, 0};
}  // namespace

void arm_wait_test(int which, uint32_t limit_ns) { t_wait_test_ns[which] = limit_ns; }

uint32_t take_wait_test(int which, int* withhold) {
  const uint32_t t = t_wait_test_ns[which];
  t_wait_test_ns[which] = 0;
  *withhold = t != 0;
  return t != 0 ? t : static_cast<uint32_t>(kWaitTimeoutNs);
}

bool make_tmap_dqacc(CUtensorMap* map, void* base, int planes, int rows, int D) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tmap_encoder();
  if (enc == nullptr) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(rows),
                        static_cast<cuuint64_t>(planes)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 4,
                           static_cast<cuuint64_t>(rows) * D * 4};
  cuuint32_t box[3] = {32, 128, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool make_tmap_bf16(CUtensorMap* map, const void* base, int planes, int rows, int D) {
  return make_tmap_16bit(map, base, planes, rows, D, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16);
}

bool make_tmap_out(CUtensorMap* map, const void* base, int planes, int rows, int D,
                   CUtensorMapDataType type) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tmap_encoder();
  if (enc == nullptr) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(rows),
                        static_cast<cuuint64_t>(planes)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2,
                           static_cast<cuuint64_t>(rows) * D * 2};
  cuuint32_t box[3] = {32, 32, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, type, 3, const_cast<void*>(base), dims,
                   strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                   CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool make_tmap_f16(CUtensorMap* map, const void* base, int planes, int rows, int D) {
  return make_tmap_16bit(map, base, planes, rows, D, CU_TENSOR_MAP_DATA_TYPE_FLOAT16);
}

}  // namespace bd

using namespace bd;

extern "C" {

const char* bd_status_string(int status) {
  switch (status) {
    case BD_OK: return "ok";
    case BD_ERR_INVALID_ARG: return "invalid argument";
    case BD_ERR_UNSUPPORTED: return "unsupported configuration";
    case BD_ERR_CUDA: return "CUDA error";
    case BD_ERR_TIMEOUT: return "device wait timed out";
    case BD_ERR_WORKSPACE: return "plan or workspace buffer too small";
    default: return "unknown status";
  }
}

int bd_version(void) { return 200; }

int bd_doc_ids_from_cu_seqlens(const int32_t* cu, const int32_t* row_ptr, int B, int S,
                               int32_t* doc_ids, int32_t* dev_status, bd_stream_t stream) {
  if (cu == nullptr || row_ptr == nullptr || doc_ids == nullptr || B < 1 || S < 1)
    return BD_ERR_INVALID_ARG;
  if (B > 65535) return BD_ERR_UNSUPPORTED;
  return launch_doc_ids(cu, row_ptr, B, S, doc_ids, dev_status, stream) == cudaSuccess
             ? BD_OK
             : BD_ERR_CUDA;
}

int bd_segment_cu_seqlens(const int32_t* doc_ids, int B, int S, int32_t* seg, int32_t* seg_ids,
                          int32_t* nseg, bd_stream_t stream) {
  if (doc_ids == nullptr || seg == nullptr || seg_ids == nullptr || nseg == nullptr || B < 1 ||
      S < 1)
    return BD_ERR_INVALID_ARG;
  if (S >= (1 << 30)) return BD_ERR_UNSUPPORTED;
  return launch_segments(doc_ids, B, S, seg, seg_ids, nseg, stream) == cudaSuccess ? BD_OK
                                                                                  : BD_ERR_CUDA;
}

int bd_doc_ids_from_seq_lens(const int32_t* seq_lens, int B, int ndocs, int S, int padding_value,
                             int32_t* doc_ids, int32_t* dev_status, bd_stream_t stream) {
  if (doc_ids == nullptr || B < 1 || S < 1 || ndocs < 0 || (ndocs > 0 && seq_lens == nullptr))
    return BD_ERR_INVALID_ARG;
  if (S >= (1 << 30) || B > 65535 || ndocs > kMaxDocsPerRow) return BD_ERR_UNSUPPORTED;
  return launch_doc_ids_from_lens(seq_lens, B, ndocs, S, padding_value, doc_ids, dev_status,
                                  stream) == cudaSuccess
             ? BD_OK
             : BD_ERR_CUDA;
}

int bd_position_ids_from_doc_ids(const int32_t* doc_ids, int B, int S, int32_t* positions,
                                 uint8_t* keep, bd_stream_t stream) {
  if (doc_ids == nullptr || positions == nullptr || keep == nullptr || B < 1 || S < 1)
    return BD_ERR_INVALID_ARG;
  if (S >= (1 << 30)) return BD_ERR_UNSUPPORTED;
  return launch_position_ids(doc_ids, B, S, positions, keep, stream) == cudaSuccess ? BD_OK
                                                                                    : BD_ERR_CUDA;
}

int bd_validate_document_positions(const uint8_t* keep, const int32_t* positions, int B, int S,
                                   int32_t* first_bad, int32_t* dev_status, bd_stream_t stream) {
  if (keep == nullptr || positions == nullptr || first_bad == nullptr || B < 1 || S < 1)
    return BD_ERR_INVALID_ARG;
  if (S >= (1 << 30)) return BD_ERR_UNSUPPORTED;
  return launch_validate_positions(keep, positions, B, S, first_bad, dev_status, stream) ==
                 cudaSuccess
             ? BD_OK
             : BD_ERR_CUDA;
}

int bd_kv_needed_range(const int32_t* seg, const int32_t* seg_ids, const int32_t* nseg, int B,
                       int S, int L, int seq_start, int32_t* range, int32_t* shard_rows,
                       bd_stream_t stream) {
  if (seg == nullptr || seg_ids == nullptr || nseg == nullptr || range == nullptr || B < 1 ||
      S < 1 || L < 1 || seq_start < 0 || static_cast<long long>(seq_start) + L > S)
    return BD_ERR_INVALID_ARG;
  if (S >= (1 << 30)) return BD_ERR_UNSUPPORTED;
  return launch_kv_range(seg, seg_ids, nseg, B, S, L, seq_start, range, shard_rows, stream) ==
                 cudaSuccess
             ? BD_OK
             : BD_ERR_CUDA;
}

size_t bd_attn_plan_size(int B, int Hq, int Hkv, int L, int S) {
  if (B < 1 || Hq < 1 || Hkv < 1 || L < 1 || S < 1) return 0;
  return plan_layout(B, Hq, Hkv, L, S).total;
}

int bd_attn_plan(const int32_t* seg, const int32_t* seg_ids, const int32_t* nseg, int B, int Hq,
                 int Hkv, int L, int S, int seq_start, void* plan, size_t plan_bytes,
                 bd_stream_t stream) {
  if (seg == nullptr || seg_ids == nullptr || nseg == nullptr || plan == nullptr)
    return BD_ERR_INVALID_ARG;
  if (B < 1 || Hq < 1 || Hkv < 1 || L < 1 || S < 1 || seq_start < 0 ||
      static_cast<long long>(seq_start) + L > S || Hq % Hkv != 0)
    return BD_ERR_INVALID_ARG;
  if (!aligned(plan, 256)) return BD_ERR_INVALID_ARG;
  if (S >= (1 << 30) || B > 65535) return BD_ERR_UNSUPPORTED;
  int st = check_plan_lists(B, Hq, Hkv, L, S);
  if (st != BD_OK) return st;
  if (plan_bytes < plan_layout(B, Hq, Hkv, L, S).total) return BD_ERR_WORKSPACE;
  return launch_plan(seg, seg_ids, nseg, B, Hq, Hkv, L, S, seq_start, plan, stream) == cudaSuccess
             ? BD_OK
             : BD_ERR_CUDA;
}

size_t bd_attn_fwd_planned_workspace_size(int B, int Hkv, int S, int D) {
  if (B < 1 || Hkv < 1 || S < 1 || D < 1) return 0;
  return align256(2 * (size_t)B * Hkv * S * D);
}

size_t bd_attn_workspace_size(int B, int Hq, int Hkv, int L, int S, int D) {
  if (B < 1 || Hq < 1 || Hkv < 1 || L < 1 || S < 1 || D < 1) return 0;
  return ws_layout(B, Hq, Hkv, L, S, D).total;
}

}  // extern "C"

namespace bd {
namespace {

// Argument checks shared by every attention entry point.
int check_attn_args(const void* q, const void* k, const void* v, int B, int Hq, int Hkv, int L,
                    int S, int D, int seq_start, int enable_gqa) {
  if (q == nullptr || k == nullptr || v == nullptr) return BD_ERR_INVALID_ARG;
  int st = check_dims(B, Hq, Hkv, L, S, D, seq_start, enable_gqa);
  if (st != BD_OK) return st;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16)) return BD_ERR_INVALID_ARG;
  return check_plan_lists(B, Hq, Hkv, L, S);
}

// The forward kernel on a built plan, v16 holding (or about to hold) the fp16 copy of v.
int fwd_run(const void* q, const void* k, int B, int Hq, int Hkv, int L, int S, int D,
            int seq_start, float scale, void* plan, void* v16, void* out, float* lse,
            void* out16, const DropoutArgs& drop, int32_t* dev_status, int sms,
            cudaStream_t stream, void* acc = nullptr, size_t acc_bytes = 0,
            uint32_t* acc_flags = nullptr) {
  AttnDims d = resolve(B, Hq, Hkv, L, S, D, seq_start, scale);
  d.drop = drop;
  CUtensorMap tq, tk, tv, to, to16;
  // (without out16 its map is never used; it then describes out)
  if (!make_tmap_out(&to, out, B * Hq, L, D, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) ||
      !make_tmap_out(&to16, out16 != nullptr ? out16 : out, B * Hq, L, D,
                     CU_TENSOR_MAP_DATA_TYPE_FLOAT16))
    return BD_ERR_CUDA;
  if (!make_tmap_bf16(&tq, q, B * Hq, L, D) || !make_tmap_bf16(&tk, k, B * Hkv, S, D) ||
      !make_tmap_f16(&tv, v16, B * Hkv, S, D))
    return BD_ERR_CUDA;
  return launch_fwd(tq, tk, tv, to, to16, d, plan, out, out16, lse, dev_status, sms, stream, acc,
                    acc_bytes, acc_flags) == cudaSuccess
             ? BD_OK
             : BD_ERR_CUDA;
}

int fwd_planned_impl(const void* q, const void* k, const void* v, int B, int Hq, int Hkv, int L,
                     int S, int D, int seq_start, float scale, int enable_gqa, void* plan,
                     size_t plan_bytes, void* out, float* lse, void* out16, void* workspace,
                     size_t workspace_bytes, const DropoutArgs& drop, int32_t* dev_status,
                     cudaStream_t stream) {
  if (plan == nullptr || out == nullptr || lse == nullptr || workspace == nullptr)
    return BD_ERR_INVALID_ARG;
  if (out16 != nullptr && !aligned(out16, 16)) return BD_ERR_INVALID_ARG;
  int st = check_attn_args(q, k, v, B, Hq, Hkv, L, S, D, seq_start, enable_gqa);
  if (st != BD_OK) return st;
  if (!aligned(out, 16) || !aligned(lse, 4) || !aligned(plan, 256) || !aligned(workspace, 256))
    return BD_ERR_INVALID_ARG;
  if (plan_bytes < plan_layout(B, Hq, Hkv, L, S).total) return BD_ERR_WORKSPACE;
  if (workspace_bytes < bd_attn_fwd_planned_workspace_size(B, Hkv, S, D)) return BD_ERR_WORKSPACE;
  const int sms = num_sms_current();
  if (sms <= 0) return BD_ERR_CUDA;
  // the P V product reads v through its fp16 copy in the workspace
  if (launch_v_to_f16(v, workspace, (long long)B * Hkv * S * D, sms, stream) != cudaSuccess)
    return BD_ERR_CUDA;
  return fwd_run(q, k, B, Hq, Hkv, L, S, D, seq_start, scale, plan, workspace, out, lse, out16,
                 drop, dev_status, sms, stream);
}

WsTag ws_tag(int B, int Hq, int Hkv, int L, int S, int D, int seq_start, const void* out,
             const float* lse, const int32_t* cu, const int32_t* row_ptr) {
  WsTag t{};
  t.cu = reinterpret_cast<uintptr_t>(cu);
  t.row_ptr = reinterpret_cast<uintptr_t>(row_ptr);
  t.flags = 0;
  t.magic = kWsMagic;
  t.B = B;
  t.Hq = Hq;
  t.Hkv = Hkv;
  t.L = L;
  t.S = S;
  t.D = D;
  t.seq_start = seq_start;
  t.out = reinterpret_cast<uintptr_t>(out);
  t.lse = reinterpret_cast<uintptr_t>(lse);
  return t;
}

int fwd_cu_impl(const void* q, const void* k, const void* v, int B, int Hq, int Hkv, int L,
                int S, int D, const int32_t* cu, const int32_t* row_ptr, int seq_start,
                float scale, int enable_gqa, void* out, float* lse, void* workspace,
                size_t workspace_bytes, const DropoutArgs& drop, int32_t* dev_status,
                cudaStream_t stream) {
  if (cu == nullptr || row_ptr == nullptr || out == nullptr || lse == nullptr ||
      workspace == nullptr)
    return BD_ERR_INVALID_ARG;
  int st = check_attn_args(q, k, v, B, Hq, Hkv, L, S, D, seq_start, enable_gqa);
  if (st != BD_OK) return st;
  if (!aligned(out, 16) || !aligned(lse, 4) || !aligned(workspace, 256)) return BD_ERR_INVALID_ARG;
  const WsLayout wl = ws_layout(B, Hq, Hkv, L, S, D);
  if (workspace_bytes < wl.total) return BD_ERR_WORKSPACE;
  const int sms = num_sms_current();
  if (sms <= 0) return BD_ERR_CUDA;
  char* ws = static_cast<char*>(workspace);
  const PlanPtrs pp = plan_ptrs(ws + wl.plan_off, B, Hq, Hkv, L, S, seq_start);
  WsTag* hdr = reinterpret_cast<WsTag*>(ws + wl.hdr);
  if (launch_prep_fwd(cu, row_ptr, pp, ws_tag(B, Hq, Hkv, L, S, D, seq_start, out, lse, cu, row_ptr),
                      hdr, v, ws + wl.v16, (long long)B * Hkv * S * D, dev_status, sms,
                      stream) != cudaSuccess)
    return BD_ERR_CUDA;
  // the forward's idle warps zero the backward's dq accumulator in the same workspace
  return fwd_run(q, k, B, Hq, Hkv, L, S, D, seq_start, scale, ws + wl.plan_off, ws + wl.v16, out,
                 lse, ws + wl.out16, drop, dev_status, sms, stream,
                 ws + wl.bwd_off + wl.bwd.dqacc, sizeof(float) * (size_t)B * Hq * L * D,
                 &hdr->flags);
}

// The backward stages on a plan; `prep` set for the single-call form.
int bwd_run(const void* q, const void* k, const void* v, const void* out, const void* out16,
            const float* lse, const void* dout, int B, int Hq, int Hkv, int L, int S, int D,
            int seq_start, float scale, void* plan, void* dq, void* dk, void* dv, void* bwd_ws,
            const DropoutArgs& drop, int32_t* dev_status, int stages, const BwdPrep* prep,
            cudaStream_t stream) {
  AttnDims d = resolve(B, Hq, Hkv, L, S, D, seq_start, scale);
  d.drop = drop;
  const BwdLayout wl = bwd_layout(B, Hq, Hkv, L, S, D);
  CUtensorMap tq, tk, tv, tdo, tdq;
  char* ws = static_cast<char*>(bwd_ws);
  if (!make_tmap_bf16(&tq, q, B * Hq, L, D) || !make_tmap_bf16(&tk, k, B * Hkv, S, D) ||
      !make_tmap_bf16(&tv, v, B * Hkv, S, D) || !make_tmap_bf16(&tdo, dout, B * Hq, L, D) ||
      !make_tmap_dqacc(&tdq, ws + wl.dqacc, B * Hq, L, D))
    return BD_ERR_CUDA;
  const int sms = num_sms_current();
  if (sms <= 0) return BD_ERR_CUDA;
  return launch_bwd(tq, tk, tv, tdo, tdq, d, plan, out, out16, lse, dout, dq, dk, dv, bwd_ws,
                    dev_status, stages, sms, stream, prep) == cudaSuccess
             ? BD_OK
             : BD_ERR_CUDA;
}

int check_bwd_ptrs(const void* out, const float* lse, const void* dout, void* dq, void* dk,
                   void* dv, void* workspace) {
  if (out == nullptr || lse == nullptr || dout == nullptr || dq == nullptr || dk == nullptr ||
      dv == nullptr || workspace == nullptr)
    return BD_ERR_INVALID_ARG;
  if (!aligned(out, 16) || !aligned(dout, 16) || !aligned(dq, 16) || !aligned(dk, 16) ||
      !aligned(dv, 16) || !aligned(lse, 4) || !aligned(workspace, 256))
    return BD_ERR_INVALID_ARG;
  return BD_OK;
}

int bwd_planned_impl(const void* q, const void* k, const void* v, const void* out,
                     const void* out16, const float* lse, const void* dout, int B, int Hq,
                     int Hkv, int L, int S, int D, int seq_start, float scale, int enable_gqa,
                     void* plan, size_t plan_bytes, void* dq, void* dk, void* dv,
                     void* workspace, size_t workspace_bytes, const DropoutArgs& drop,
                     int32_t* dev_status, cudaStream_t stream) {
  if (plan == nullptr) return BD_ERR_INVALID_ARG;
  if (out16 != nullptr && !aligned(out16, 16)) return BD_ERR_INVALID_ARG;
  int st = check_attn_args(q, k, v, B, Hq, Hkv, L, S, D, seq_start, enable_gqa);
  if (st != BD_OK) return st;
  st = check_bwd_ptrs(out, lse, dout, dq, dk, dv, workspace);
  if (st != BD_OK) return st;
  if (!aligned(plan, 256)) return BD_ERR_INVALID_ARG;
  if (plan_bytes < plan_layout(B, Hq, Hkv, L, S).total) return BD_ERR_WORKSPACE;
  if (workspace_bytes < bwd_layout(B, Hq, Hkv, L, S, D).total) return BD_ERR_WORKSPACE;
  return bwd_run(q, k, v, out, out16, lse, dout, B, Hq, Hkv, L, S, D, seq_start, scale, plan, dq,
                 dk, dv, workspace, drop, dev_status, kBwdPrepare | kBwdMain | kBwdFinish,
                 nullptr, stream);
}

int bwd_cu_impl(const void* q, const void* k, const void* v, const void* out, const float* lse,
                const void* dout, int B, int Hq, int Hkv, int L, int S, int D,
                const int32_t* cu, const int32_t* row_ptr, int seq_start, float scale,
                int enable_gqa, void* dq, void* dk, void* dv, void* workspace,
                size_t workspace_bytes, const DropoutArgs& drop, int32_t* dev_status, int stages,
                cudaStream_t stream) {
  if (cu == nullptr || row_ptr == nullptr) return BD_ERR_INVALID_ARG;
  if (stages <= 0 || stages > (kBwdPrepare | kBwdMain | kBwdFinish)) return BD_ERR_INVALID_ARG;
  int st = check_attn_args(q, k, v, B, Hq, Hkv, L, S, D, seq_start, enable_gqa);
  if (st != BD_OK) return st;
  st = check_bwd_ptrs(out, lse, dout, dq, dk, dv, workspace);
  if (st != BD_OK) return st;
  const WsLayout wl = ws_layout(B, Hq, Hkv, L, S, D);
  if (workspace_bytes < wl.total) return BD_ERR_WORKSPACE;
  char* ws = static_cast<char*>(workspace);
  BwdPrep prep{};
  prep.cu = cu;
  prep.row_ptr = row_ptr;
  prep.pp = plan_ptrs(ws + wl.plan_off, B, Hq, Hkv, L, S, seq_start);
  prep.hdr = reinterpret_cast<WsTag*>(ws + wl.hdr);
  prep.expect = ws_tag(B, Hq, Hkv, L, S, D, seq_start, out, lse, cu, row_ptr);
  return bwd_run(q, k, v, out, ws + wl.out16, lse, dout, B, Hq, Hkv, L, S, D, seq_start, scale,
                 ws + wl.plan_off, dq, dk, dv, ws + wl.bwd_off, drop, dev_status, stages, &prep,
                 stream);
}

}  // namespace
}  // namespace bd

extern "C" {

int bd_attn_fwd(const void* q, const void* k, const void* v, int B, int Hq, int Hkv, int L, int S,
                int D, const int32_t* cu_seqlens, const int32_t* row_ptr, int seq_start,
                float scale, int enable_gqa, void* out, float* lse, void* workspace,
                size_t workspace_bytes, int32_t* dev_status, bd_stream_t stream) {
  return fwd_cu_impl(q, k, v, B, Hq, Hkv, L, S, D, cu_seqlens, row_ptr, seq_start, scale,
                     enable_gqa, out, lse, workspace, workspace_bytes, DropoutArgs{}, dev_status,
                     stream);
}

int bd_attn_bwd(const void* q, const void* k, const void* v, const void* out, const float* lse,
                const void* dout, int B, int Hq, int Hkv, int L, int S, int D,
                const int32_t* cu_seqlens, const int32_t* row_ptr, int seq_start, float scale,
                int enable_gqa, void* dq, void* dk, void* dv, void* workspace,
                size_t workspace_bytes, int32_t* dev_status, bd_stream_t stream) {
  return bwd_cu_impl(q, k, v, out, lse, dout, B, Hq, Hkv, L, S, D, cu_seqlens, row_ptr,
                     seq_start, scale, enable_gqa, dq, dk, dv, workspace, workspace_bytes,
                     DropoutArgs{}, dev_status, kBwdPrepare | kBwdMain | kBwdFinish, stream);
}

int bd_attn_bwd_stages(const void* q, const void* k, const void* v, const void* out,
                       const float* lse, const void* dout, int B, int Hq, int Hkv, int L, int S,
                       int D, const int32_t* cu_seqlens, const int32_t* row_ptr, int seq_start,
                       float scale, int enable_gqa, void* dq, void* dk, void* dv,
                       void* workspace, size_t workspace_bytes, int32_t* dev_status, int stages,
                       bd_stream_t stream) {
  return bwd_cu_impl(q, k, v, out, lse, dout, B, Hq, Hkv, L, S, D, cu_seqlens, row_ptr,
                     seq_start, scale, enable_gqa, dq, dk, dv, workspace, workspace_bytes,
                     DropoutArgs{}, dev_status, stages, stream);
}

int bd_attn_fwd_dropout(const void* q, const void* k, const void* v, int B, int Hq, int Hkv,
                        int L, int S, int D, const int32_t* cu_seqlens, const int32_t* row_ptr,
                        int seq_start, float scale, int enable_gqa, void* out, float* lse,
                        void* workspace, size_t workspace_bytes, double dropout_p, uint64_t seed,
                        uint32_t offset, int32_t* dev_status, bd_stream_t stream) {
  DropoutArgs drop;
  const int st = make_dropout(dropout_p, seed, offset, &drop);
  if (st != BD_OK) return st;
  return fwd_cu_impl(q, k, v, B, Hq, Hkv, L, S, D, cu_seqlens, row_ptr, seq_start, scale,
                     enable_gqa, out, lse, workspace, workspace_bytes, drop, dev_status, stream);
}

int bd_attn_bwd_dropout(const void* q, const void* k, const void* v, const void* out,
                        const float* lse, const void* dout, int B, int Hq, int Hkv, int L, int S,
                        int D, const int32_t* cu_seqlens, const int32_t* row_ptr, int seq_start,
                        float scale, int enable_gqa, void* dq, void* dk, void* dv,
                        void* workspace, size_t workspace_bytes, double dropout_p, uint64_t seed,
                        uint32_t offset, int32_t* dev_status, bd_stream_t stream) {
  DropoutArgs drop;
  const int st = make_dropout(dropout_p, seed, offset, &drop);
  if (st != BD_OK) return st;
  return bwd_cu_impl(q, k, v, out, lse, dout, B, Hq, Hkv, L, S, D, cu_seqlens, row_ptr,
                     seq_start, scale, enable_gqa, dq, dk, dv, workspace, workspace_bytes, drop,
                     dev_status, kBwdPrepare | kBwdMain | kBwdFinish, stream);
}

int bd_attn_fwd_planned(const void* q, const void* k, const void* v, int B, int Hq, int Hkv,
                        int L, int S, int D, int seq_start, float scale, int enable_gqa,
                        void* plan, size_t plan_bytes, void* out, float* lse, void* out16,
                        void* workspace, size_t workspace_bytes, int32_t* dev_status,
                        bd_stream_t stream) {
  return fwd_planned_impl(q, k, v, B, Hq, Hkv, L, S, D, seq_start, scale, enable_gqa, plan,
                          plan_bytes, out, lse, out16, workspace, workspace_bytes,
                          DropoutArgs{}, dev_status, stream);
}

int bd_attn_fwd_dropout_planned(const void* q, const void* k, const void* v, int B, int Hq,
                                int Hkv, int L, int S, int D, int seq_start, float scale,
                                int enable_gqa, void* plan, size_t plan_bytes, void* out,
                                float* lse, void* out16, void* workspace, size_t workspace_bytes,
                                double dropout_p, uint64_t seed, uint32_t offset,
                                int32_t* dev_status, bd_stream_t stream) {
  DropoutArgs drop;
  const int st = make_dropout(dropout_p, seed, offset, &drop);
  if (st != BD_OK) return st;
  return fwd_planned_impl(q, k, v, B, Hq, Hkv, L, S, D, seq_start, scale, enable_gqa, plan,
                          plan_bytes, out, lse, out16, workspace, workspace_bytes, drop,
                          dev_status, stream);
}

size_t bd_attn_bwd_planned_workspace_size(int B, int Hq, int Hkv, int L, int S, int D) {
  if (B < 1 || Hq < 1 || Hkv < 1 || L < 1 || S < 1 || D < 1) return 0;
  return bwd_layout(B, Hq, Hkv, L, S, D).total;
}

int bd_attn_bwd_planned(const void* q, const void* k, const void* v, const void* out,
                        const void* out16, const float* lse, const void* dout, int B, int Hq,
                        int Hkv, int L, int S, int D, int seq_start, float scale, int enable_gqa,
                        void* plan, size_t plan_bytes, void* dq, void* dk, void* dv,
                        void* workspace, size_t workspace_bytes, int32_t* dev_status,
                        bd_stream_t stream) {
  return bwd_planned_impl(q, k, v, out, out16, lse, dout, B, Hq, Hkv, L, S, D, seq_start, scale,
                          enable_gqa, plan, plan_bytes, dq, dk, dv, workspace, workspace_bytes,
                          DropoutArgs{}, dev_status, stream);
}

int bd_attn_bwd_dropout_planned(const void* q, const void* k, const void* v, const void* out,
                                const void* out16, const float* lse, const void* dout, int B,
                                int Hq, int Hkv, int L, int S, int D, int seq_start, float scale,
                                int enable_gqa, void* plan, size_t plan_bytes, void* dq,
                                void* dk, void* dv, void* workspace, size_t workspace_bytes,
                                double dropout_p, uint64_t seed, uint32_t offset,
                                int32_t* dev_status, bd_stream_t stream) {
  DropoutArgs drop;
  const int st = make_dropout(dropout_p, seed, offset, &drop);
  if (st != BD_OK) return st;
  return bwd_planned_impl(q, k, v, out, out16, lse, dout, B, Hq, Hkv, L, S, D, seq_start, scale,
                          enable_gqa, plan, plan_bytes, dq, dk, dv, workspace, workspace_bytes,
                          drop, dev_status, stream);
}

int bd_test_arm_wait_timeout(int which, unsigned int limit_us) {
  if ((which != kWaitTestFwd && which != kWaitTestBwd) || limit_us < 1 || limit_us > 2000000u)
    return BD_ERR_INVALID_ARG;
  arm_wait_test(which, limit_us * 1000u);
  return BD_OK;
}

int bd_get_device_status(const int32_t* dev_status, int32_t* host_status, bd_stream_t stream) {
  if (dev_status == nullptr || host_status == nullptr) return BD_ERR_INVALID_ARG;
  if (cudaMemcpyAsync(host_status, dev_status, sizeof(int32_t), cudaMemcpyDeviceToHost, stream) !=
      cudaSuccess)
    return BD_ERR_CUDA;
  return cudaStreamSynchronize(stream) == cudaSuccess ? BD_OK : BD_ERR_CUDA;
}

}  // extern "C"
