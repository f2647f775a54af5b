/*
 * bd_attn.h -- C ABI of the GB300 (sm_103a) block-diagonal causal attention
 * library for packed sequences (libbd_attn.so).
 *
 * The operation is the one described on the NeMo Automodel API reference page
 * "nemo_automodel.components.distributed.blockdiag_cp", function
 * cp_blockdiag_sdpa: local queries [B, Hq, L, D] attend the delivered keys and
 * values [B, Hkv, S, D] under a per-document causal mask rebuilt from document
 * ids, so documents packed into one row never attend across a boundary.  The
 * document ids and their segments follow the page
 * "nemo_automodel.components.models.glm5_next.cp" (doc_ids_from_cu_seqlens,
 * segment_cu_seqlens, _PAD_DOC_ID = 0).  Queries may be a contiguous
 * interval [seq_start, seq_start + L) of the row (Glm5NextPackedContext
 * .seq_start on the same page), as a context-parallel rank sees them.
 *
 * Conventions for every entry point:
 *  - All tensor pointers are DEVICE pointers owned by the caller.  The library
 *    never allocates, frees or synchronises; every call only enqueues work on
 *    `stream` (a cudaStream_t; NULL = the legacy default stream) and returns.
 *  - Tensors are dense, row-major, with the shapes given below; bf16 data is
 *    passed as `const void*` / `void*` (IEEE bfloat16, 2 bytes).  q, k, v,
 *    out, dout, dq, dk, dv must be 16-byte aligned.
 *  - The return value is a bd_status_t.  Host-side argument errors return
 *    BD_ERR_INVALID_ARG / BD_ERR_UNSUPPORTED / BD_ERR_WORKSPACE before any
 *    work is enqueued.  A failed launch returns BD_ERR_CUDA.  Errors found on
 *    the device (invalid cu_seqlens, a wait that timed out) are written to the
 *    caller's `dev_status` word (int32, device memory, may be NULL); the
 *    first error of a call is kept.  bd_get_device_status() reads it back.
 *  - Document id 0 marks padding.  A query in a padding segment attends
 *    nothing: its output row is 0, its log-sum-exp -inf, its dq row 0.  Keys
 *    that no query of the call attends get dk = dv = 0.
 */
#ifndef BD_ATTN_H
#define BD_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* bd_stream_t; /* identical to cudaStream_t */

typedef enum {
  BD_OK = 0,
  BD_ERR_INVALID_ARG = 1, /* bad shape, pointer, alignment or cu_seqlens */
  BD_ERR_UNSUPPORTED = 2, /* valid but not implemented (e.g. head dim not 64/128) */
  BD_ERR_CUDA = 3,        /* a CUDA runtime call or launch failed */
  BD_ERR_TIMEOUT = 4,     /* a device-side wait gave up (reported via dev_status) */
  BD_ERR_WORKSPACE = 5    /* plan or workspace buffer too small */
} bd_status_t;

/* Human-readable text for a status code (static storage, never NULL). */
const char* bd_status_string(int status);

/* Library ABI version (major * 100 + minor): 200. */
int bd_version(void);

/*
 * Document ids from cumulative boundaries (page
 * "nemo_automodel.components.models.glm5_next.cp", doc_ids_from_cu_seqlens,
 * and _PAD_DOC_ID = 0).
 *   cu       int32, the B rows' boundary lists concatenated.  Row b's list is
 *            cu[row_ptr[b] .. row_ptr[b+1]-1]: n_b + 1 entries, starting at 0,
 *            non-decreasing, last entry <= S.  Zero-length documents allowed.
 *   row_ptr  int32 [B+1], row_ptr[0] = 0, row_ptr[b+1] - row_ptr[b] >= 1.
 *   doc_ids  int32 [B, S] output: position p of row b gets d + 1 when
 *            cu_b[d] <= p < cu_b[d+1], and 0 (padding) when p >= cu_b[n_b].
 * A row whose list breaks the rules above gets all ids 0 and
 * BD_ERR_INVALID_ARG in *dev_status.
 */
int bd_doc_ids_from_cu_seqlens(const int32_t* cu, const int32_t* row_ptr, int B, int S,
                               int32_t* doc_ids, int32_t* dev_status, bd_stream_t stream);

/*
 * Segment boundaries of each row (page
 * "nemo_automodel.components.models.glm5_next.cp", segment_cu_seqlens):
 * the maximal runs of equal ids, padding runs included, covering the row.
 *   doc_ids  int32 [B, S].
 *   seg      int32 [B, S+1] output: row b's boundaries are
 *            seg[b*(S+1) + 0 .. nseg[b]], seg[..0] = 0, seg[..nseg[b]] = S.
 *   seg_ids  int32 [B, S] output: seg_ids[b*S + k] = id carried by run k.
 *   nseg     int32 [B] output: number of runs of row b.
 * Entries past a row's count are left untouched.
 */
int bd_segment_cu_seqlens(const int32_t* doc_ids, int B, int S, int32_t* seg, int32_t* seg_ids,
                          int32_t* nseg, bd_stream_t stream);

/*
 * Document ids from per-document lengths (page
 * "nemo_automodel.components.models.glm5_next.cp", doc_ids_from_seq_lens:
 * lengths [batch, documents] padded with padding_value, default -1000).
 *   seq_lens       int32 [B, ndocs]; entries equal to padding_value are not
 *                  documents and take no number; the others are numbered
 *                  1..n in order (a zero-length document takes its number).
 *   ndocs          0 .. 8192 (larger: BD_ERR_UNSUPPORTED).
 *   doc_ids        int32 [B, S] output; positions past the last document are 0.
 * A negative length other than padding_value, or a row total above S, zeroes
 * that row and records BD_ERR_INVALID_ARG in *dev_status (first error wins).
 */
int bd_doc_ids_from_seq_lens(const int32_t* seq_lens, int B, int ndocs, int S, int padding_value,
                             int32_t* doc_ids, int32_t* dev_status, bd_stream_t stream);

/*
 * Document positions and validity from document ids (page
 * "nemo_automodel.components.models.inkling2.context_parallel",
 * unpack_row_layout: integer positions and a padding mask [batch, sequence],
 * padding decided from the document layout, never from token ids).
 *   doc_ids    int32 [B, S]; a document is a maximal run of equal non-zero ids.
 *   positions  int32 [B, S] output: 0, 1, 2, ... along each document; 0 on padding.
 *   keep       uint8 [B, S] output: 1 on document tokens, 0 on padding.
 */
int bd_position_ids_from_doc_ids(const int32_t* doc_ids, int B, int S, int32_t* positions,
                                 uint8_t* keep, bd_stream_t stream);

/*
 * Document-position check (page
 * "nemo_automodel.components.models.inkling2.context_parallel",
 * validate_document_positions: unit increments inside documents, zero at a
 * new document; a shard may begin partway through a document; a gap cannot
 * resume an old one).  Among the kept tokens of a row, in order: the first
 * may carry any position >= 0; a later one must carry 0, or its
 * predecessor's position + 1 when it directly follows the predecessor; after
 * a gap it must carry 0.
 *   keep       uint8 [B, S] (non-zero = valid token).
 *   positions  int32 [B, S].
 *   first_bad  int32 [B] output: first offending column of each row, or -1.
 * Any offending row also records BD_ERR_INVALID_ARG in *dev_status.
 */
int bd_validate_document_positions(const uint8_t* keep, const int32_t* positions, int B, int S,
                                   int32_t* first_bad, int32_t* dev_status, bd_stream_t stream);

/*
 * Key/value rows the local queries need (page
 * "nemo_automodel.components.distributed.blockdiag_cp", cp_blockdiag_sdpa:
 * K/V delivered by all-gather "or a needed-only halo/a2a exchange").  The
 * local queries [seq_start, seq_start + L) attend, under the per-document
 * causal mask, exactly the rows [lo, hi): lo = start of the segment of the
 * first non-padding local query, hi = one past the last non-padding local
 * query; lo = hi = seq_start when every local query is padding.
 *   seg, seg_ids, nseg  as written by bd_segment_cu_seqlens for [B, S].
 *   range       int32 [B, 2] output: (lo, hi) of each row.
 *   shard_rows  int32 [B, ceil(S / L)] output, or NULL: rows of [lo, hi) in
 *               each shard [r L, min((r + 1) L, S)) of the row (the counts an
 *               all-to-all-v of shards of L rows would move).
 */
int bd_kv_needed_range(const int32_t* seg, const int32_t* seg_ids, const int32_t* nseg, int B,
                       int S, int L, int seq_start, int32_t* range, int32_t* shard_rows,
                       bd_stream_t stream);

/*
 * Attention plan: per-row mask bounds, the non-empty tile ranges of every
 * query block (forward) and key tile (backward), and both work lists in the
 * order the kernels take them (the forward's longest first; the backward's by
 * document, largest first, each document's tiles together and longest first).
 * This is the "varlen metadata precompute" that the page
 * "nemo_automodel.components.distributed.blockdiag_cp" names as an internal
 * detail.  Built on the device from the output of bd_segment_cu_seqlens,
 * with no host synchronisation.
 *   seg, seg_ids, nseg  as written by bd_segment_cu_seqlens for [B, S].
 *   Hq, Hkv             head counts (the plan's forward blocks depend on
 *                       whether Hq / Hkv is even).
 *   L, seq_start        query rows are global positions seq_start .. +L-1.
 *   plan                device buffer of bd_attn_plan_size() bytes, 256-byte
 *                       aligned, used by bd_attn_fwd_planned / bd_attn_bwd_planned, which must
 *                       be given the same B, Hq, Hkv, L, S, seq_start.  It also
 *                       holds the work counters those kernels take units from
 *                       (in the lists' order) and leave at zero when they finish, so
 *                       one plan must not serve two launches that overlap in
 *                       time (use one plan per stream).
 * Returns BD_ERR_UNSUPPORTED when B * ceil(L/128) or B * ceil(S/128)
 * exceeds 16384.
 */
size_t bd_attn_plan_size(int B, int Hq, int Hkv, int L, int S);
int bd_attn_plan(const int32_t* seg, const int32_t* seg_ids, const int32_t* nseg, int B, int Hq,
                 int Hkv, int L, int S, int seq_start, void* plan, size_t plan_bytes,
                 bd_stream_t stream);

/*
 * Forward pass in one call (page
 * "nemo_automodel.components.distributed.blockdiag_cp", cp_blockdiag_sdpa:
 * output [B, Hq, L, D] for the local rows, the mask "rebuilt from the
 * document ids"; ids as doc_ids_from_cu_seqlens on the page
 * "nemo_automodel.components.models.glm5_next.cp").
 *   q            bf16 [B, Hq, L, D]; query i sits at global position seq_start+i.
 *   k, v         bf16 [B, Hkv, S, D], the full key/value row.
 *   D            64 or 128 (else BD_ERR_UNSUPPORTED).
 *   cu_seqlens,  each row's cumulative document boundaries, as for
 *   row_ptr      bd_doc_ids_from_cu_seqlens (both device arrays; row_ptr is
 *                required for every B).  The document of a position and its
 *                bounds are found from them on the device; a row whose list
 *                is invalid is treated as all padding and BD_ERR_INVALID_ARG
 *                goes to *dev_status.
 *   seq_start    0 <= seq_start, seq_start + L <= S.
 *   scale        softmax scale; a value <= 0 or not finite means D^-0.5
 *                ("None -> D**-0.5" on the page).
 *   enable_gqa   must be non-zero when Hq != Hkv (Hq a multiple of Hkv);
 *                query head h reads key/value head h / (Hq / Hkv).
 *   out          bf16 [B, Hq, L, D] output.
 *   lse          fp32 [B, Hq, L] output: natural-log log-sum-exp of the
 *                scaled scores of each row (-inf for padding rows).
 *   workspace    device scratch of bd_attn_workspace_size() bytes, 256-byte
 *                aligned, owned by the caller.  The call keeps there the
 *                attention plan (mask bounds and ordered work lists),
 *                an fp16 copy of v (the P V product runs with fp16 operands:
 *                v must lie within the fp16 range, |x| <= 65504), and an
 *                fp16 copy of the result O for the backward, with a record
 *                of the shapes and of out and lse.  Too small:
 *                BD_ERR_WORKSPACE.
 * Validation on the host: B, Hq, Hkv, L, S >= 1, Hq % Hkv == 0, the interval
 * inside the row, 16-byte aligned q, k, v, out, and B * ceil(L/128),
 * B * ceil(S/128) <= 16384 (else BD_ERR_UNSUPPORTED).
 */
size_t bd_attn_workspace_size(int B, int Hq, int Hkv, int L, int S, int D);
int bd_attn_fwd(const void* q, const void* k, const void* v, int B, int Hq, int Hkv, int L, int S,
                int D, const int32_t* cu_seqlens, const int32_t* row_ptr, int seq_start,
                float scale, int enable_gqa, void* out, float* lse, void* workspace,
                size_t workspace_bytes, int32_t* dev_status, bd_stream_t stream);

/*
 * Backward pass in one call: gradients of sum(out * dout) (the autograd
 * backward of bd_attn_fwd).  Same arguments as bd_attn_fwd plus
 *   out, lse     the forward's outputs for these inputs.
 *   dout         bf16 [B, Hq, L, D].
 *   dq           bf16 [B, Hq, L, D] output.
 *   dk, dv       bf16 [B, Hkv, S, D] outputs, summed over the query heads of
 *                each group; fully overwritten (rows no query attends are 0).
 *   workspace    bd_attn_workspace_size() bytes.  The plan is rebuilt from
 *                the boundaries.  Delta_i = <dO_i, O_i> takes O from the fp16
 *                copy the forward kept in the workspace when the workspace
 *                still records this out and lse with these shapes (pass the
 *                workspace of the forward call, untouched in between, for
 *                full precision); otherwise from the bf16 out.
 * The dq accumulation uses floating-point atomics, so dq may differ in the
 * last bits between runs; dk and dv are deterministic.  All five products
 * (K Q^T, V dO^T, P^T dO, dS^T Q, dS K) take bf16 operands with fp32
 * accumulation; P and dS = P (dP - Delta) are rounded to bf16 for them.
 */
int bd_attn_bwd(const void* q, const void* k, const void* v, const void* out, const float* lse,
                const void* dout, int B, int Hq, int Hkv, int L, int S, int D,
                const int32_t* cu_seqlens, const int32_t* row_ptr, int seq_start, float scale,
                int enable_gqa, void* dq, void* dk, void* dv, void* workspace,
                size_t workspace_bytes, int32_t* dev_status, bd_stream_t stream);

/*
 * bd_attn_bwd in separately launchable stages (same arguments plus a bit
 * mask), meant for timing one stage at a time.  Bit 1: the plan from the
 * boundaries, per-row terms -lse log2 e and -Delta, and the zeroed fp32 dq
 * accumulator (one launch).  Bit 2: the main kernel (dk, dv written; dq
 * accumulated in the workspace).  Bit 4: dq = bf16(scale * accumulator).
 * The stages must run in this order on the same workspace; bd_attn_bwd is
 * stages = 7.
 */
int bd_attn_bwd_stages(const void* q, const void* k, const void* v, const void* out,
                       const float* lse, const void* dout, int B, int Hq, int Hkv, int L, int S,
                       int D, const int32_t* cu_seqlens, const int32_t* row_ptr, int seq_start,
                       float scale, int enable_gqa, void* dq, void* dk, void* dv,
                       void* workspace, size_t workspace_bytes, int32_t* dev_status, int stages,
                       bd_stream_t stream);

/*
 * Forward and backward with attention dropout (page
 * "nemo_automodel.components.distributed.blockdiag_cp", cp_blockdiag_sdpa's
 * dropout_p, read as torch scaled_dot_product_attention's: dropout acts on
 * the normalised attention weights and kept ones are scaled up; p is taken
 * on a 16-bit grain, below).
 * Same arguments and results as bd_attn_fwd / bd_attn_bwd plus
 *   dropout_p    in [0, 1) (else BD_ERR_INVALID_ARG); 0 is no dropout.
 *   seed         64-bit key of the generator.
 *   offset       32-bit stream offset (a different offset draws a different
 *                mask under the same seed, e.g. one per layer or step).
 * The mask is a pure function of (seed, offset, batch row b, query head h,
 * query position t, key position j): weight (t, j) of plane b * Hq + h is
 * dropped iff its 16-bit value is below floor(p * 2^16), where the value is
 * the low (j even) or high (j odd) half of word (j & 7) >> 1 of
 * Philox4x32-10 (Salmon et al., SC'11) at counter (j >> 3, t, b * Hq + h,
 * offset) under key (seed mod 2^32, seed >> 32).  The drop probability is
 * thus p' = floor(p * 2^16) / 2^16 (p rounded down to the 16-bit grain;
 * below 2^-16 nothing is dropped) and kept weights are scaled by
 * 1 / (1 - p'), so the output's expectation is the undropped one.
 * t is the global position
 * (seq_start + i), so query intervals of one row draw the same mask as the
 * whole row, and the backward regenerates the forward's mask from the same
 * (seed, offset) with nothing stored in between.  lse stays the log-sum-exp
 * of the undropped scores; out is the dropped output.  The backward must be
 * given the forward's dropout_p, seed and offset.
 */
int bd_attn_fwd_dropout(const void* q, const void* k, const void* v, int B, int Hq, int Hkv,
                        int L, int S, int D, const int32_t* cu_seqlens, const int32_t* row_ptr,
                        int seq_start, float scale, int enable_gqa, void* out, float* lse,
                        void* workspace, size_t workspace_bytes, double dropout_p, uint64_t seed,
                        uint32_t offset, int32_t* dev_status, bd_stream_t stream);
int bd_attn_bwd_dropout(const void* q, const void* k, const void* v, const void* out,
                        const float* lse, const void* dout, int B, int Hq, int Hkv, int L, int S,
                        int D, const int32_t* cu_seqlens, const int32_t* row_ptr, int seq_start,
                        float scale, int enable_gqa, void* dq, void* dk, void* dv,
                        void* workspace, size_t workspace_bytes, double dropout_p, uint64_t seed,
                        uint32_t offset, int32_t* dev_status, bd_stream_t stream);

/*
 * Lower-level forms on a plan from bd_attn_plan, for callers that hold
 * document ids rather than boundaries (padding anywhere in a row, ids that
 * repeat after a gap: the mask then follows the segments of the ids).  Same
 * operation, arguments and results as the calls above, with
 *   plan         from bd_attn_plan with the same B, Hq, Hkv, L, S, seq_start.
 *   out16        forward: optional fp16 [B, Hq, L, D] output (NULL to skip):
 *                the fp32 result O rounded to fp16 (11 significant bits
 *                against out's 8), without the dropout factor 1 / (1 - p),
 *                so that its entries lie within the range of v; backward:
 *                that output of the forward with the same dropout_p (Delta
 *                from it, times 1 / (1 - p)), or NULL (Delta from out).
 *   workspace    forward: bd_attn_fwd_planned_workspace_size() bytes (the
 *                fp16 copy of v); backward:
 *                bd_attn_bwd_planned_workspace_size() bytes (the fp32 dq
 *                accumulator and per-row terms); 256-byte aligned.
 * Dropout arguments as above.
 */
size_t bd_attn_fwd_planned_workspace_size(int B, int Hkv, int S, int D);
int bd_attn_fwd_planned(const void* q, const void* k, const void* v, int B, int Hq, int Hkv,
                        int L, int S, int D, int seq_start, float scale, int enable_gqa,
                        void* plan, size_t plan_bytes, void* out, float* lse, void* out16,
                        void* workspace, size_t workspace_bytes, int32_t* dev_status,
                        bd_stream_t stream);
int bd_attn_fwd_dropout_planned(const void* q, const void* k, const void* v, int B, int Hq,
                                int Hkv, int L, int S, int D, int seq_start, float scale,
                                int enable_gqa, void* plan, size_t plan_bytes, void* out,
                                float* lse, void* out16, void* workspace, size_t workspace_bytes,
                                double dropout_p, uint64_t seed, uint32_t offset,
                                int32_t* dev_status, bd_stream_t stream);
size_t bd_attn_bwd_planned_workspace_size(int B, int Hq, int Hkv, int L, int S, int D);
int bd_attn_bwd_planned(const void* q, const void* k, const void* v, const void* out,
                        const void* out16, const float* lse, const void* dout, int B, int Hq,
                        int Hkv, int L, int S, int D, int seq_start, float scale, int enable_gqa,
                        void* plan, size_t plan_bytes, void* dq, void* dk, void* dv,
                        void* workspace, size_t workspace_bytes, int32_t* dev_status,
                        bd_stream_t stream);
int bd_attn_bwd_dropout_planned(const void* q, const void* k, const void* v, const void* out,
                                const void* out16, const float* lse, const void* dout, int B,
                                int Hq, int Hkv, int L, int S, int D, int seq_start, float scale,
                                int enable_gqa, void* plan, size_t plan_bytes, void* dq,
                                void* dk, void* dv, void* workspace, size_t workspace_bytes,
                                double dropout_p, uint64_t seed, uint32_t offset,
                                int32_t* dev_status, bd_stream_t stream);

/*
 * The backward pass without any caller-provided scratch, for callers that
 * cannot allocate device memory: for example code running inside a host
 * runtime that reserves all GPU memory when it starts and forbids further
 * allocation (a cudaMalloc can synchronise the device, stall other work, or
 * fail once memory is fragmented).  The pages describe no such variant; it
 * is an addition of this library.
 *
 * Same arguments and results as bd_attn_bwd_planned, minus the workspace.
 * The scratch is a fixed array of BD_NOALLOC_SCRATCH_BYTES (16 MiB) that the
 * library image places on every GPU that loads it, held until the process
 * exits.  Problems whose bd_attn_bwd_planned_workspace_size() exceeds that return
 * BD_ERR_WORKSPACE before anything is launched.  Nothing is allocated.
 *  - The first call on each device looks up the array's device address (with
 *    that device current) and caches it; make that first call before any
 *    stream capture begins.
 *  - Every call uses the same array and leaves its contents behind; each call
 *    clears what must start at zero itself.  Calls whose GPU work overlaps in
 *    time (two streams, or several threads) race on the array and give wrong
 *    results: serialise them.
 */
#define BD_NOALLOC_SCRATCH_BYTES (16u << 20)
int bd_attn_bwd_noalloc(const void* q, const void* k, const void* v, const void* out,
                        const void* out16, const float* lse, const void* dout, int B, int Hq,
                        int Hkv, int L, int S, int D, int seq_start, float scale, int enable_gqa,
                        void* plan, size_t plan_bytes, void* dq, void* dk, void* dv,
                        int32_t* dev_status, bd_stream_t stream);

/*
 * Test hook for the bounded device-side waits (the pages have no counterpart;
 * it exists to test this library's failure path).  Every wait of the
 * forward and backward kernels gives up after 2 s, records BD_ERR_TIMEOUT in
 * dev_status, lets the rest of the CTA stop, waits (bounded) for its own
 * copies and tensor-core work in flight, frees its tensor memory and returns,
 * so the context stays usable.  This call makes the next launch of one
 * kernel from the calling host thread exercise that path on purpose: its
 * producer publishes its first work unit but never loads that unit's first
 * tile, and its waits give up after limit_us microseconds instead of 2 s.
 *   which      1: the forward kernel (bd_attn_fwd*), 2: the backward main
 *              kernel (bd_attn_bwd*, stage 2).
 *   limit_us   1 .. 2000000.
 * The request is used by that one launch and then dropped; its results are
 * not valid (the status says BD_ERR_TIMEOUT).  Returns BD_ERR_INVALID_ARG for
 * other arguments.
 */
int bd_test_arm_wait_timeout(int which, unsigned int limit_us);

/*
 * Copy the device status word to *host_status after the work already queued
 * on `stream` finishes (this call synchronises `stream`; no other entry point
 * does).  Returns BD_OK or BD_ERR_CUDA.
 */
int bd_get_device_status(const int32_t* dev_status, int32_t* host_status, bd_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* BD_ATTN_H */
