// Backward pass of block-diagonal causal attention: gradients of
// sum(out * dout) for cp_blockdiag_sdpa (page
// "nemo_automodel.components.distributed.blockdiag_cp"), written from the
// softmax derivative: Delta_i = <dO_i, o_i>, P = exp(S - lse),
// dS = P * (dP - Delta), dq = scale dS K, dk = scale dS^T Q, dv = P^T dO.
//
// Kernels:
//  bwd_pre    -Delta and -lse (log2 units) per row, zero the fp32 dq accumulator
//  bd_bwd     persistent; one work unit = one 128-key tile of one K/V head,
//             looping over the G query heads of the group and the query tiles
//             the plan marks non-empty.  Per iteration (tcgen05, TMEM):
//               S^T = K Q^T, dP^T = V dO^T          (cols 256, 384)
//               P^T back into TMEM; dS -> smem (both bf16)
//               dV += P^T dO, dK += dS^T Q          (cols 128, 0)
//               dQ = dS K                           (cols 384, once dS is formed)
//             four warps read dQ out of TMEM, stage it in shared memory
//             and adds it into the fp32 accumulator with TMA reductions;
//             dK, dV leave once per unit.
//  bwd_dq     dq = bf16(scale * accumulator)
#include "bd_pre_dev.cuh"

namespace bd {

namespace {

// 20 warps: producer, MMA, dQ reduction issuer, one idle warp, two P/dS
// warpgroups and two dQ reader warpgroups (64 columns of dQ each).
constexpr int kThreads = 640;

template <int D>
struct BwdCfg {
  static constexpr int TILE = 128 * D * 2;  // bytes of a 128-row bf16 tile
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = TILE;
  static constexpr int OFF_Q = 2 * TILE;              // [2 stages]
  // dO_i is read only by dP^T_i (the end of iteration i-1) and dV_i (the start
  // of iteration i), so one buffer suffices: dO_{i+1} loads while dS_i is
  // formed.  The 32 KB this saves hold the dQ staging buffer.
  static constexpr int OFF_DO = OFF_Q + 2 * TILE;
  static constexpr int OFF_DS = OFF_DO + TILE;        // 128 keys x 128 queries bf16
  static constexpr int OFF_STG = OFF_DS + 32768;      // 64 columns of dQ_i in fp32
  static constexpr int OFF_LSED = OFF_STG + 32768;    // [2 stages] 128 x float2
  static constexpr int OFF_BAR = OFF_LSED + 2048;
  static constexpr int SMEM = OFF_BAR + 320;  // barriers, TMEM slot, abort flag, work ring
  // All five products take bf16 operands straight from the inputs (P and dS
  // rounded to bf16), fp32 accumulation in TMEM.
  static constexpr uint32_t IDESC_S = make_idesc(128, 128, 0, 0, 1);   // S^T = K Q^T
  static constexpr uint32_t IDESC_DP = make_idesc(128, 128, 0, 0, 1);  // dP^T = V dO^T
  static constexpr uint32_t IDESC_DV = make_idesc(128, D, 0, 1, 1);    // dV += P^T dO
  static constexpr uint32_t IDESC_DK = make_idesc(128, D, 0, 1, 1);    // dK += dS^T Q
  static constexpr uint32_t IDESC_DQ = make_idesc(128, D, 1, 1, 1);    // dQ = dS K
};

struct BwdParams {
  int B, Hq, Hkv, L, S, seq_start, G, NKT, Spad, Lq, n_units;
  float scale_log2, scale;
  const int32_t* kend;
  const int32_t* bwd_range;
  const int32_t* bwd_order;
  // negated so that the P and dS phases add them with paired fp32 arithmetic
  const float* nlse2;   // -lse * log2(e) per query row, -inf where the row attends nothing
  const float* ndelta;  // -Delta = -<dO, O> per query row
  float* dqacc;
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  int32_t* status;
  int* ctr;  // work counters in the plan: [next unit, finished CTAs]
  int* aborts;  // CTAs of the launch that gave up a wait (in the plan)
  uint32_t* acc_flags;  // optional: kAccZeroed is cleared (the accumulator now holds sums)
  uint32_t wait_limit_ns;  // bound of every device-side wait
  int withhold;            // test only: the producer withholds the first K/V load
  DropoutArgs drop;
};

struct BUnit {
  int b, g, kt, qt_lo, nq, n_it;
};

__device__ __forceinline__ BUnit decode_bunit(const BwdParams& p, int w) {
  BUnit u;
  const int e = w / p.Hkv;
  u.g = w % p.Hkv;
  const int ktl = p.bwd_order[e];
  u.b = ktl / p.NKT;
  u.kt = ktl % p.NKT;
  u.qt_lo = p.bwd_range[2 * ktl];
  u.nq = p.bwd_range[2 * ktl + 1] - u.qt_lo + 1;
  u.n_it = u.nq > 0 ? u.nq * p.G : 0;
  return u;
}

// Iteration i of a unit: query head g*G + i/nq, query tile counted down from
// the last one the key tile reaches.  Every unit of a document and head then
// starts on the same tile and the units running side by side walk the same
// Q/dO tiles and dq-accumulator rows at about the same time, which keeps them
// in L2.
__device__ __forceinline__ int unit_qtile(const BUnit& u, int i) {
  return u.qt_lo + u.nq - 1 - i % u.nq;
}

// Dropout keep bits of one key row against 64 consecutive queries (bit c:
// the query at global position t0 + c), for a thread whose key is `key`.
// The element (query t, key j) keeps iff the 16-bit half j & 1 of word
// (j & 7) >> 1 of Philox4x32-10 at counter (j >> 3, t, plane, offset)
// reaches the threshold.  The eight lanes of an octet hold the eight keys of
// one counter, so each lane draws the blocks of 8 of the queries (one block
// serves all eight keys) and the octet then exchanges the bits: byte g of
// lane a holds the eight keys' bits of query 8 g + a.
__device__ __forceinline__ uint64_t keep_bits64(int key, uint32_t t0, uint32_t plane,
                                                const DropoutArgs& d, int lane) {
  const int a = lane & 7;
  const uint32_t thr = d.threshold;
  uint64_t bytes = 0;
#pragma unroll
  for (int g = 0; g < 8; ++g) {
    const uint4 w = philox4x32_10(static_cast<uint32_t>(key) >> 3, t0 + 8 * g + a, plane,
                                  d.offset, d.rk);
    const uint32_t n = static_cast<uint32_t>((w.x & 0xffffu) >= thr) |
                       (static_cast<uint32_t>((w.x >> 16) >= thr) << 1) |
                       (static_cast<uint32_t>((w.y & 0xffffu) >= thr) << 2) |
                       (static_cast<uint32_t>((w.y >> 16) >= thr) << 3) |
                       (static_cast<uint32_t>((w.z & 0xffffu) >= thr) << 4) |
                       (static_cast<uint32_t>((w.z >> 16) >= thr) << 5) |
                       (static_cast<uint32_t>((w.w & 0xffffu) >= thr) << 6) |
                       (static_cast<uint32_t>((w.w >> 16) >= thr) << 7);
    bytes |= static_cast<uint64_t>(n) << (8 * g);
  }
  uint64_t out = 0;
#pragma unroll
  for (int src = 0; src < 8; ++src) {
    const uint64_t x = __shfl_sync(0xffffffffu, bytes, (lane & ~7) | src);
    out |= ((x >> a) & 0x0101010101010101ull) << src;  // key a's bit of query 8 g + src
  }
  return out;
}

__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity, int32_t* status) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > kWaitTimeoutNs) {
      set_status(status, BD_ERR_TIMEOUT);
      return;
    }
  }
}

__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}

}  // namespace

// ------------------------------------------------------------------ preprocess

// One thread per 8 elements of a query row: -Delta, -lse in log2 units and the
// zeroed dq accumulator (bwd_pre_rows in bd_pre_dev.cuh).
template <int D>
__global__ void __launch_bounds__(256) bwd_pre_kernel(
    const __nv_bfloat16* __restrict__ out, const __half* __restrict__ out16, float o16_scale,
    const __nv_bfloat16* __restrict__ dout, const float* __restrict__ lse, int planes, int L,
    int Lq, float* __restrict__ nlse2o, float* __restrict__ ndeltao, float* __restrict__ dqacc) {
  bwd_pre_rows<D>((long long)blockIdx.x * blockDim.x + threadIdx.x, out, out16, o16_scale, dout,
                  lse, planes, L, Lq, nlse2o, ndeltao, dqacc);
}

template <int D>
__global__ void __launch_bounds__(256) bwd_dq_kernel(const float* __restrict__ dqacc,
                                                     __nv_bfloat16* __restrict__ dq,
                                                     long long n8, float scale) {
  const long long t = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= n8) return;
  // Both streams are touched once: load and store them evict-first, so that
  // the accumulator lines the main kernel left in L2 are not pushed out by
  // dq before this pass reaches them (28.7 us against 30.7 on 8,192 tokens,
  // 32 heads, D = 128).
  const float4* src = reinterpret_cast<const float4*>(dqacc) + 2 * t;
  const float4 a = __ldcs(src), b = __ldcs(src + 1);
  uint4 o;
  o.x = pack_bf16x2(a.x * scale, a.y * scale);
  o.y = pack_bf16x2(a.z * scale, a.w * scale);
  o.z = pack_bf16x2(b.x * scale, b.y * scale);
  o.w = pack_bf16x2(b.z * scale, b.w * scale);
  __stcs(reinterpret_cast<uint4*>(dq) + t, o);
}

// ------------------------------------------------------------------ main kernel
//
// Per iteration i (query tile x head of the unit's group), TMEM columns:
//   dK [0,128)  dV [128,256)  S^T -> P^T [256,384)  dP^T -> dQ [384,512)
// (at D = 64 dQ has columns of its own, [64,128), beside dK)
// Tensor-core order (one thread):
//   dV += P^T_i dO_i | S^T_{i+1} | dK += dS^T_i Q_i | dQ_i = dS_i K | dP^T_{i+1}
// so that the P/dS work overlaps MMAs: dS_i is formed while dV_i and S^T_{i+1}
// run, P_{i+1} while dK_i, dQ_i and dP^T_{i+1} run.  dS_i lives only in
// shared memory (the A operand of both dK_i and dQ_i), so dQ_i can take the
// dP^T columns as soon as dS_i is formed.  (dK_i goes first: the dQ read-out
// then starts later but finds the staging buffer free sooner.)  Two warpgroups share
// that work by query columns (64 each), which puts two such warps on every
// scheduler.  Each keeps P_i between its two phases as the bf16 pairs it
// hands to the dV MMA (32 registers) and forms dS = P (dP - Delta) in fp32
// from them.

// kDrop: attention dropout (p.drop).  With the mask M regenerated from the
// counters the forward used: dV = rp (P o M)^T dO, where the P^T tile carries
// P o M and rp = 1 / (1 - p) joins dV's epilogue; dS = P o (rp M o dP - Delta),
// Delta = <dO, O> of the dropped output.
template <int D, bool kDrop>
__global__ void __launch_bounds__(kThreads, 1)
    bd_bwd_kernel(const __grid_constant__ CUtensorMap tmap_q,
                  const __grid_constant__ CUtensorMap tmap_k,
                  const __grid_constant__ CUtensorMap tmap_v,
                  const __grid_constant__ CUtensorMap tmap_do,
                  const __grid_constant__ CUtensorMap tmap_dq, const __grid_constant__ BwdParams p) {
  using C = BwdCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* kv_full = bars + 0;
  uint64_t* kv_empty = bars + 1;
  uint64_t* st_full = bars + 2;   // [2]
  uint64_t* st_empty = bars + 4;  // [2]
  uint64_t* s_full = bars + 6;
  uint64_t* dp_full = bars + 7;
  uint64_t* p_full = bars + 8;
  uint64_t* ds_full = bars + 9;
  uint64_t* dq_full = bars + 10;
  uint64_t* dq_empty = bars + 11;
  uint64_t* dkdv_full = bars + 12;
  uint64_t* drain = bars + 13;
  // stg_full[s]: a 16 KB box of dQ_i is in staging slot s (the issuer alone
  // waits, box by box).  stg_read[2 s + g]: the TMA has read the box that
  // reader group g put in slot s; one phase per iteration each, so a reader
  // that waits for the other group's box cannot be two phases behind (its own
  // previous box in the slot may still be unread).
  uint64_t* stg_full = bars + 14;  // [2]
  uint64_t* stg_read = bars + 16;  // [4]
  uint64_t* do_full = bars + 20;   // dO_i landed
  uint64_t* do_empty = bars + 21;  // dV_i done: the dO buffer may be refilled
  // ds_half (D = 64): the first 32 queries of each P/dS group's dS_i are in
  // shared memory (the dK k-steps over those queries can start)
  uint64_t* ds_half = bars + 22;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 23);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);  // + the wait limit
  WorkRing* ring = reinterpret_cast<WorkRing*>(bars + 25);
  static_assert(25 * 8 + sizeof(WorkRing) <= C::SMEM - C::OFF_BAR, "barrier area too small");
  static_assert(C::SMEM <= 232448, "shared memory over the per-block limit");

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    abort_flag[0] = 0;
    abort_flag[1] = static_cast<int>(p.wait_limit_ns);
    if ((smem_u32(smem) & 1023u) != 0) {
      set_status(p.status, BD_ERR_CUDA);
      *abort_flag = 1;
    }
    mbar_init(kv_full, 1);
    mbar_init(kv_empty, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(st_full + s, 1);
      mbar_init(st_empty + s, 1);
    }
    mbar_init(s_full, 1);
    mbar_init(dp_full, 1);
    mbar_init(p_full, 256);
    mbar_init(ds_full, 256);
    mbar_init(ds_half, 256);
    mbar_init(dq_full, 1);
    mbar_init(dq_empty, 2 * D);  // the reader threads that hold dQ columns
    mbar_init(dkdv_full, 1);
    mbar_init(drain, 1);
    for (int s = 0; s < 2; ++s) mbar_init(stg_full + s, 128);
    for (int s = 0; s < 4; ++s) mbar_init(stg_read + s, 1);
    mbar_init(do_full, 1);
    mbar_init(do_empty, 1);
    ring_init(ring, 18);  // MMA thread, reduction issuer, 8 P/dS warps, 8 dQ readers
    fence_mbar_init();
    prefetch_tmap(&tmap_q);
    prefetch_tmap(&tmap_k);
    prefetch_tmap(&tmap_v);
    prefetch_tmap(&tmap_do);
    prefetch_tmap(&tmap_dq);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const bool aborted_at_start = *abort_flag != 0;

  if (warp == 0 && !aborted_at_start) {
    // ------------------------------------------------------------ producer + work queue
    if (lane == 0) {
      uint32_t kv_u = 0, st_it = 0, do_it = 0, kq = 0;  // fills issued: K/V, Q stages, dO
      for (;;) {
        int w;
        if (!ring_publish(ring, kq++, p.ctr, p.n_units, abort_flag, p.status, w) || w < 0) break;
        const BUnit u = decode_bunit(p, w);
        if (u.n_it <= 0) continue;
        // test of the bounded waits: the unit is published but its K/V never
        // arrive, so the MMA thread's wait for them runs out
        if (p.withhold) break;
        if (!mbar_wait(kv_empty, (kv_u & 1) ^ 1, abort_flag, p.status)) break;
        mbar_arrive_expect_tx(kv_full, 2 * C::TILE);
        const int kvplane = u.b * p.Hkv + u.g;
        for (int j = 0; j < D / 64; ++j) {
          tma_load_3d(smem + C::OFF_K + j * 16384, &tmap_k, kv_full, 64 * j, u.kt * kBN, kvplane);
          tma_load_3d(smem + C::OFF_V + j * 16384, &tmap_v, kv_full, 64 * j, u.kt * kBN, kvplane);
        }
        ++kv_u;
        bool ok = true;
        for (int i = 0; i < u.n_it; ++i) {
          const int h = u.g * p.G + i / u.nq;
          const int qt = unit_qtile(u, i);
          const int st = st_it & 1;
          ok = mbar_wait(st_empty + st, ((st_it >> 1) & 1) ^ 1, abort_flag, p.status);
          if (!ok) break;
          mbar_arrive_expect_tx(st_full + st, C::TILE + 1024);
          const int qplane = u.b * p.Hq + h;
          for (int j = 0; j < D / 64; ++j)
            tma_load_3d(smem + C::OFF_Q + st * C::TILE + j * 16384, &tmap_q, st_full + st, 64 * j,
                        qt * kBM, qplane);
          const size_t ro = (size_t)qplane * p.Lq + qt * kBM;
          bulk_load(smem + C::OFF_LSED + st * 1024, p.nlse2 + ro, 512, st_full + st);
          bulk_load(smem + C::OFF_LSED + st * 1024 + 512, p.ndelta + ro, 512, st_full + st);
          ++st_it;
          // dO_i after dV_{i-1}; Q_{i+1} (next round) waits for dK_{i-1}, which follows dV_{i-1}
          ok = mbar_wait(do_empty, (do_it & 1) ^ 1, abort_flag, p.status);
          if (!ok) break;
          mbar_arrive_expect_tx(do_full, C::TILE);
          for (int j = 0; j < D / 64; ++j)
            tma_load_3d(smem + C::OFF_DO + j * 16384, &tmap_do, do_full, 64 * j, qt * kBM, qplane);
          ++do_it;
        }
        if (!ok) break;
      }
      if (kv_u > 0) drain_wait(kv_full, (kv_u - 1) & 1, p.status);
      for (int st = 0; st < 2; ++st) {
        if (st_it > static_cast<uint32_t>(st)) {
          const uint32_t last = st_it - 1 - ((st_it - 1 - st) & 1);
          drain_wait(st_full + st, (last >> 1) & 1, p.status);
        }
      }
      if (do_it > 0) drain_wait(do_full, (do_it - 1) & 1, p.status);
    }
    __syncwarp();
  } else if (warp == 1 && !aborted_at_start) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t sk = smem_u32(smem + C::OFF_K);
      const uint32_t sv = smem_u32(smem + C::OFF_V);
      const uint32_t sq0 = smem_u32(smem + C::OFF_Q);
      const uint32_t sdo0 = smem_u32(smem + C::OFF_DO);
      const uint32_t sds = smem_u32(smem + C::OFF_DS);
      const uint32_t tDK = tmem, tDV = tmem + 128, tS = tmem + 256, tDP = tmem + 384;
      // At D = 64 dQ has columns of its own ([64, 128), beside dK), so dP^T_{i+1}
      // need not wait for dQ_i to be read out; at D = 128 it shares dP^T's.
      constexpr bool kOwnDQ = D == 64;
      const uint32_t tDQ = kOwnDQ ? tmem + 64 : tDP;
      // D[128 keys, 128 queries] = A[keys, D] (K-major) * B[queries, D]^T (K-major)
      // Each operand's descriptor is built once per product and stepped by a
      // constant per instruction (sdesc_add), and every step but the first
      // accumulates through a folded predicate: this thread's instruction
      // count per tcgen05.mma stays low.
      auto issue_kmajor = [&](uint32_t d, uint32_t a, uint32_t b, uint32_t idesc) {
        const uint64_t ad = make_sdesc_sw128(a, 16, 1024), bd = make_sdesc_sw128(b, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
          if (kk == 0)
            mma_ss(d, ad, bd, idesc, 0);
          else
            mma_ss_acc(d, sdesc_add(ad, off), sdesc_add(bd, off), idesc);
        }
      };
      // D[keys, D] (+)= A[tmem, keys x 128 queries] * B[queries, D] (MN-major smem).
      // A's 16-bit pairs for queries [0, 64) sit at columns [0, 32) of its
      // 128-column region and those for [64, 128) at [64, 96) (each P/dS
      // warpgroup packs into the first half of its own columns).
      auto issue_ts = [&](uint32_t d, uint32_t a_tmem, uint32_t b, bool acc, uint32_t idesc) {
        const uint64_t bd = make_sdesc_sw128(b, 16384, 1024);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          if (ks == 0)
            mma_ts(d, a_tmem, bd, idesc, acc);
          else
            mma_ts_acc(d, a_tmem + ks * 8 + (ks >= 4 ? 32 : 0), sdesc_add(bd, ks * 2048), idesc);
        }
      };
      // dK[keys, D] += dS^T[keys, queries] * Q[queries, D]: the dS tile (key rows,
      // queries contiguous) is the K-major A operand, Q the MN-major B operand.
      // Issued in two halves: part 0 takes the k-steps over queries [0, 32) and
      // [64, 96) (the first 32 queries of each P/dS group, ready at ds_half at
      // D = 64), part 1 the rest; the first instruction of part 0 sets or
      // accumulates.  At D = 64, where the P/dS warps and this thread bound
      // the period together, starting part 0 early took causal64k's backward
      // from 82.7 to 81.7 ms; at D = 128 it cost short documents ~1%, so there
      // all eight k-steps go in order once the whole of dS is in.
      // part < 0: all eight k-steps in order.
      auto issue_dk = [&](uint32_t b, bool acc, int part) {
        const uint64_t ad = make_sdesc_sw128(sds, 16, 1024), bd = make_sdesc_sw128(b, 16384, 1024);
#pragma unroll
        for (int j = 0; j < (part < 0 ? 8 : 4); ++j) {
          // 0..7, or 0,1,4,5 (part 0) or 2,3,6,7 (part 1)
          const int kk = part < 0 ? j : (j >> 1) * 4 + part * 2 + (j & 1);
          const uint64_t a = sdesc_add(ad, (kk >> 2) * 16384 + (kk & 3) * 32);
          if (part <= 0 && j == 0)
            mma_ss(tDK, a, bd, C::IDESC_DK, acc);
          else
            mma_ss_acc(tDK, a, sdesc_add(bd, kk * 2048), C::IDESC_DK);
        }
      };
      // dQ[queries, D] = dS[queries, keys] (MN-major smem) * K[keys, D] (MN-major smem)
      auto issue_dq = [&]() {
        const uint64_t ad = make_sdesc_sw128(sds, 16384, 1024);
        const uint64_t bd = make_sdesc_sw128(sk, 16384, 1024);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          if (ks == 0)
            mma_ss(tDQ, ad, bd, C::IDESC_DQ, 0);
          else
            mma_ss_acc(tDQ, sdesc_add(ad, ks * 2048), sdesc_add(bd, ks * 2048), C::IDESC_DQ);
        }
      };
      uint32_t kv_u = 0, st_it = 0, it_g = 0, kq = 0;
      bool ok = true;
      while (ok) {
        int w;
        if (!ring_take(ring, kq++, abort_flag, p.status, w) || w < 0) break;
        const BUnit u = decode_bunit(p, w);
        if (u.n_it <= 0) continue;
        ok = mbar_wait(kv_full, kv_u & 1, abort_flag, p.status);
        if (!ok) break;
        int st = st_it & 1;
        ok = mbar_wait(st_full + st, (st_it >> 1) & 1, abort_flag, p.status);
        if (!ok) break;
        tc_fence_after();
        issue_kmajor(tS, sk, sq0 + st * C::TILE, C::IDESC_S);
        mma_commit(s_full);
        if (!kOwnDQ && it_g > 0) {  // the previous iteration's dQ must have left the dP columns
          ok = mbar_wait(dq_empty, (it_g - 1) & 1, abort_flag, p.status);
          if (!ok) break;
        }
        ok = mbar_wait(do_full, st_it & 1, abort_flag, p.status);
        if (!ok) break;
        tc_fence_after();
        issue_kmajor(tDP, sv, sdo0, C::IDESC_DP);
        mma_commit(dp_full);
        for (int i = 0; i < u.n_it && ok; ++i) {
          const uint32_t si = st_it + i;
          st = si & 1;
          const int sn = (si + 1) & 1;
          const bool more = i + 1 < u.n_it;
          ok = mbar_wait(p_full, it_g & 1, abort_flag, p.status);
          if (!ok) break;
          tc_fence_after();
          issue_ts(tDV, tS, sdo0, i > 0, C::IDESC_DV);
          mma_commit(do_empty);  // dO_i is no longer read
          if (more) {
            ok = mbar_wait(st_full + sn, ((si + 1) >> 1) & 1, abort_flag, p.status);
            if (!ok) break;
            tc_fence_after();
            issue_kmajor(tS, sk, sq0 + sn * C::TILE, C::IDESC_S);
            mma_commit(s_full);
          }
          if constexpr (D == 64) {
            ok = mbar_wait(ds_half, it_g & 1, abort_flag, p.status);
            if (!ok) break;
            tc_fence_after();
            issue_dk(sq0 + st * C::TILE, i > 0, 0);
          }
          ok = mbar_wait(ds_full, it_g & 1, abort_flag, p.status);
          if (!ok) break;
          tc_fence_after();
          if constexpr (D == 64)
            issue_dk(sq0 + st * C::TILE, true, 1);
          else
            issue_dk(sq0 + st * C::TILE, i > 0, -1);
          mma_commit(st_empty + st);  // Q_i is no longer read after dK_i
          if (kOwnDQ && it_g > 0) {  // the previous dQ must have been read out of its columns
            ok = mbar_wait(dq_empty, (it_g - 1) & 1, abort_flag, p.status);
            if (!ok) break;
          }
          issue_dq();
          mma_commit(dq_full);
          if (more) {
            if (!kOwnDQ) {
              ok = mbar_wait(dq_empty, it_g & 1, abort_flag, p.status);
              if (!ok) break;
            }
            ok = mbar_wait(do_full, (si + 1) & 1, abort_flag, p.status);
            if (!ok) break;
            tc_fence_after();
            issue_kmajor(tDP, sv, sdo0, C::IDESC_DP);
            mma_commit(dp_full);
          }
          ++it_g;
        }
        st_it += u.n_it;
        mma_commit(kv_empty);
        mma_commit(dkdv_full);
        ++kv_u;
      }
      mma_commit(drain);
      drain_wait(drain, 0, p.status);
    }
    __syncwarp();
  } else if (warp >= 4 && warp < 12 && !aborted_at_start) {
    // ------------------------------------------------------------ P / dS warpgroups
    // Warpgroup hf (1 or 2 -> hf 0 or 1) takes the 64 queries [64 hf, 64 hf + 64)
    // of every key row; the two groups reach the same TMEM lanes (lane access
    // follows the warp's index mod 4).
    const int hf = (warp - 4) >> 2;
    const int q4 = warp & 3;
    const int r = q4 * 32 + lane;  // key row of the tile = TMEM lane
    const int c0 = 64 * hf;        // first query column of this group
    const uint32_t lane_off = static_cast<uint32_t>(q4 * 32) << 16;
    // S^T / dP^T columns of this group; P^T (bf16 pairs) goes back into the
    // first half of its S^T columns, behind the reads
    const uint32_t tS = tmem + lane_off + 256 + c0, tDP = tmem + lane_off + 384 + c0;
    const uint32_t sds_row = smem_u32(smem + C::OFF_DS) + hf * 16384 + (r >> 3) * 1024 +
                             (r & 7) * 128;
    uint32_t st_it = 0, it_g = 0, kv_u = 0, kq = 0;
    for (;;) {
      int w;
      if (!ring_take_warp(ring, kq++, abort_flag, p.status, w) || w < 0) break;
      const BUnit u = decode_bunit(p, w);
      const int key = u.kt * kBN + r;
      const size_t krow = ((size_t)(u.b * p.Hkv + u.g) * p.S + key) * D;
      // group 1 owns dK of the tile, group 2 dV
      __nv_bfloat16* const grad = (hf == 0 ? p.dk : p.dv) + krow;
      if (u.n_it <= 0) {
        if (key < p.S) {
          uint4* a = reinterpret_cast<uint4*>(grad);
#pragma unroll
          for (int c = 0; c < D / 8; ++c) a[c] = make_uint4(0, 0, 0, 0);
        }
        continue;
      }
      const int kend = p.kend[(size_t)u.b * p.Spad + key];
      bool ok = true;
      for (int i = 0; i < u.n_it; ++i) {
        const int qt = unit_qtile(u, i);
        const int st = st_it & 1;
        uint32_t keep_lo = 0xffffffffu, keep_hi = 0xffffffffu;  // dropout keep bits of the 64 columns
        if constexpr (kDrop) {
          // drawn before the S^T wait: they depend only on the positions
          const uint32_t plane = static_cast<uint32_t>(u.b * p.Hq + u.g * p.G + i / u.nq);
          const uint64_t kb = keep_bits64(
              key, static_cast<uint32_t>(p.seq_start + qt * kBM + c0), plane, p.drop, lane);
          keep_lo = static_cast<uint32_t>(kb);
          keep_hi = static_cast<uint32_t>(kb >> 32);
        }
        // ---- phase P: P^T = exp2(S^T * scale * log2 e - lse * log2 e), masked
        ok = mbar_wait_warp(s_full, it_g & 1, abort_flag, p.status);
        if (!ok) break;
        ok = mbar_wait_warp(st_full + st, (st_it >> 1) & 1, abort_flag, p.status);
        if (!ok) break;
        tc_fence_after();
        // columns c (query q0 + c) attending this key: key <= q0 + c < min(kend, end of interval)
        const int q0 = p.seq_start + qt * kBM;
        int ca = 1, cb = 0;
        if (kend > key) {
          ca = key - q0;
          cb = min(kend, p.seq_start + p.L) - q0 - 1;
        }
        const bool full = __all_sync(0xffffffffu, ca <= c0 && cb >= c0 + 63);
        uint32_t mw[2];  // allowed columns of this group's 64, 32 per word
#pragma unroll
        for (int w = 0; w < 2; ++w) {
          const int lo = max(ca - c0 - 32 * w, 0), hi = min(cb - c0 - 32 * w, 31);
          mw[w] = (lo > hi) ? 0u
                            : ((0xffffffffu >> (31 - max(hi, 0))) & (0xffffffffu << min(lo, 31)));
        }
        // the stage holds -lse*log2(e) of the tile's 128 queries, then their -Delta
        const float4* nlse4 =
            reinterpret_cast<const float4*>(smem + C::OFF_LSED + st * 1024) + (c0 >> 2);
        const float4* ndl4 = nlse4 + 32;
        const float2 sc2 = make_float2(p.scale_log2, p.scale_log2);
        uint32_t pk[32];  // P^T of this key row as bf16 pairs (the dV MMA's operand), kept for dS
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t sv[32], tmp[16];
          tmem_ld32(tS + c * 32, sv);
#pragma unroll
          for (int e = 0; e < 32; e += 4) {
            const float4 x = nlse4[(c * 32 + e) >> 2];  // -lse*log2(e) of four columns
            const float2 t01 = ffma2(make_float2(__uint_as_float(sv[e]), __uint_as_float(sv[e + 1])),
                                     sc2, make_float2(x.x, x.y));
            const float2 t23 =
                ffma2(make_float2(__uint_as_float(sv[e + 2]), __uint_as_float(sv[e + 3])), sc2,
                      make_float2(x.z, x.w));
            float p0 = fast_exp2(t01.x);
            float p1 = fast_exp2(t01.y);
            float p2 = fast_exp2(t23.x);
            float p3 = fast_exp2(t23.y);
            if (!full) {
              const uint32_t m = mw[c] >> e;
              p0 = (m & 1u) ? p0 : 0.f;
              p1 = (m & 2u) ? p1 : 0.f;
              p2 = (m & 4u) ? p2 : 0.f;
              p3 = (m & 8u) ? p3 : 0.f;
            }
            pk[c * 16 + (e >> 1)] = pack_bf16x2(p0, p1);
            pk[c * 16 + (e >> 1) + 1] = pack_bf16x2(p2, p3);
            if constexpr (kDrop) {
              // P o M for dV: a dropped weight's bf16 half becomes 0
              const uint32_t kb = (c == 0 ? keep_lo : keep_hi) >> e;
              tmp[e >> 1] = pk[c * 16 + (e >> 1)] & ((kb & 1u ? 0x0000ffffu : 0u) |
                                                     (kb & 2u ? 0xffff0000u : 0u));
              tmp[(e >> 1) + 1] = pk[c * 16 + (e >> 1) + 1] & ((kb & 4u ? 0x0000ffffu : 0u) |
                                                               (kb & 8u ? 0xffff0000u : 0u));
            }
          }
          if constexpr (!kDrop) {
#pragma unroll
            for (int e = 0; e < 16; ++e) tmp[e] = pk[c * 16 + e];
          }
          tmem_st16(tS + c * 16, tmp);
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(p_full);
        // ---- phase dS: dS = P * (dP - Delta) -> smem (the A operand of dK and dQ)
        ok = mbar_wait_warp(dp_full, it_g & 1, abort_flag, p.status);
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t dv[32];
          tmem_ld32(tDP + c * 32, dv);
          uint32_t dk[16];
#pragma unroll
          for (int e = 0; e < 32; e += 4) {
            const float4 x = ndl4[(c * 32 + e) >> 2];  // -Delta of four columns
            const uint32_t pa = pk[c * 16 + (e >> 1)], pb = pk[c * 16 + (e >> 1) + 1];
            if constexpr (kDrop) {
              // dS = P (rp M dP - Delta)
              const uint32_t kb = (c == 0 ? keep_lo : keep_hi) >> e;
              const float rp = p.drop.rp;
              const float d0 = (kb & 1u) ? fmaf(rp, __uint_as_float(dv[e]), x.x) : x.x;
              const float d1 = (kb & 2u) ? fmaf(rp, __uint_as_float(dv[e + 1]), x.y) : x.y;
              const float d2 = (kb & 4u) ? fmaf(rp, __uint_as_float(dv[e + 2]), x.z) : x.z;
              const float d3 = (kb & 8u) ? fmaf(rp, __uint_as_float(dv[e + 3]), x.w) : x.w;
              dk[e >> 1] = pack_bf16x2(__uint_as_float(pa << 16) * d0,
                                       __uint_as_float(pa & 0xffff0000u) * d1);
              dk[(e >> 1) + 1] = pack_bf16x2(__uint_as_float(pb << 16) * d2,
                                             __uint_as_float(pb & 0xffff0000u) * d3);
              continue;
            }
            // dS = P (dP + (-Delta)), in pairs
            const float2 s01 = fmul2(
                make_float2(__uint_as_float(pa << 16), __uint_as_float(pa & 0xffff0000u)),
                fadd2(make_float2(__uint_as_float(dv[e]), __uint_as_float(dv[e + 1])),
                      make_float2(x.x, x.y)));
            const float2 s23 = fmul2(
                make_float2(__uint_as_float(pb << 16), __uint_as_float(pb & 0xffff0000u)),
                fadd2(make_float2(__uint_as_float(dv[e + 2]), __uint_as_float(dv[e + 3])),
                      make_float2(x.z, x.w)));
            dk[e >> 1] = pack_bf16x2(s01.x, s01.y);
            dk[(e >> 1) + 1] = pack_bf16x2(s23.x, s23.y);
          }
          // dS (queries contiguous) into the 128-byte-swizzled tile that is the K-major
          // A operand of dK = dS^T Q and the MN-major A operand of dQ = dS K
#pragma unroll
          for (int gq = 0; gq < 4; ++gq) {
            const int cq = c * 4 + gq;  // 16-byte chunk index along this group's queries
            const uint32_t addr = sds_row + ((cq ^ (r & 7)) << 4);
            st_shared_v4(addr, dk[4 * gq], dk[4 * gq + 1], dk[4 * gq + 2], dk[4 * gq + 3]);
          }
          if (D == 64 && c == 0) {  // half of dK_i can start on these 32 queries
            fence_async_smem();
            tc_fence_before();
            mbar_arrive(ds_half);
          }
        }
        fence_async_smem();
        tc_fence_before();
        mbar_arrive(ds_full);
        ++st_it;
        ++it_g;
      }
      if (!ok) break;
      // epilogue: dK (scaled, group 1) or dV (group 2) of this key tile
      ok = mbar_wait_warp(dkdv_full, kv_u & 1, abort_flag, p.status);
      if (!ok) break;
      ++kv_u;
      tc_fence_after();
      {
        const uint32_t tsrc = tmem + lane_off + hf * 128;
        const float mul = hf == 0 ? p.scale : (kDrop ? p.drop.rp : 1.f);
        // Each 32-column chunk goes through shared memory so that four lanes
        // per row store 64 contiguous bytes, eight rows an instruction.  The
        // staging is this warp's 4 KB of its group's half of the dS tile: every
        // product of the unit has completed (dkdv_full), and only this group
        // writes that half again, in its next dS phase.  16-byte pieces are
        // swizzled by row pair, so neither side conflicts on banks; two 2 KB
        // slots alternate.
        const uint32_t stg = smem_u32(smem + C::OFF_DS) + hf * 16384 + q4 * 4096;
        const int key0 = u.kt * kBN + q4 * 32;  // the warp's first key row
        __nv_bfloat16* const gbase =
            (hf == 0 ? p.dk : p.dv) + ((size_t)(u.b * p.Hkv + u.g) * p.S + key0) * D;
        const int rr0 = lane >> 2, jj = lane & 3;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t v[32];
          tmem_ld32(tsrc + c * 32, v);
          uint32_t pk2[16];
#pragma unroll
          for (int e = 0; e < 16; ++e)
            pk2[e] = pack_bf16x2(__uint_as_float(v[2 * e]) * mul,
                                 __uint_as_float(v[2 * e + 1]) * mul);
          const uint32_t slot = stg + (c & 1) * 2048;
#pragma unroll
          for (int j = 0; j < 4; ++j)
            st_shared_v4(slot + lane * 64 + ((j ^ ((lane >> 1) & 3)) << 4), pk2[4 * j],
                         pk2[4 * j + 1], pk2[4 * j + 2], pk2[4 * j + 3]);
          __syncwarp();
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int rr = 8 * k + rr0;
            if (key0 + rr < p.S)
              *reinterpret_cast<uint4*>(gbase + (size_t)rr * D + c * 32 + jj * 8) =
                  ld_shared_v4(slot + rr * 64 + ((jj ^ ((rr >> 1) & 3)) << 4));
          }
        }
        __syncwarp();
      }
      tc_fence_before();
    }
  } else if (warp >= 12 && warp < 20 && !aborted_at_start) {
    // ------------------------------------------------------------ dQ readers
    // Reader warpgroup rg takes dQ columns [64 rg, 64 rg + 64) of every row in
    // one TMEM load (64 registers a thread) and hands the columns back at
    // once, so dP^T_{i+1} never waits for the staging.  Its columns then go
    // into the staging buffer as two 128-byte-swizzled boxes of 128 rows x 32
    // columns, box k of the call into 16 KB slot k & 1 once the TMA has read
    // the slot's previous box; warp 2 adds each box into the fp32 accumulator
    // with a TMA reduction, so the reductions never occupy the SM's load/store
    // path.
    const int rg = (warp - 12) >> 2;
    const int q4 = warp & 3;
    const int r = q4 * 32 + lane;  // query row of the tile = TMEM lane
    const uint32_t tQ =
        tmem + (static_cast<uint32_t>(q4 * 32) << 16) + (D == 64 ? 64 : 384) + 64 * rg;
    const uint32_t srow = smem_u32(smem + C::OFF_STG) + r * 128;
    constexpr uint32_t kBoxes = D / 32;  // boxes per dQ tile
    const bool active = 64 * rg < D;
    uint32_t it_g = 0, kq = 0;
    // box k of the call: slot k & 1, reader group (k mod kBoxes) / 2, and the
    // slot's previous box k - 2 was read in that box's group's iteration
    // (k - 2) / kBoxes
    auto stage_box = [&](const uint32_t (&v)[32], uint32_t k) -> bool {
      const uint32_t slot = k & 1;
      if (k >= 2) {
        const uint32_t kp = k - 2;
        const uint32_t gp = (kp % kBoxes) >> 1;
        if (!mbar_wait_warp(stg_read + 2 * slot + gp, (kp / kBoxes) & 1, abort_flag, p.status))
          return false;
      }
      const uint32_t row = srow + slot * 16384;
#pragma unroll
      for (int c = 0; c < 8; ++c)
        st_shared_v4(row + ((c ^ (r & 7)) << 4), v[c * 4], v[c * 4 + 1], v[c * 4 + 2],
                     v[c * 4 + 3]);
      fence_async_smem();
      mbar_arrive(stg_full + slot);
      return true;
    };
    for (;;) {
      int w;
      if (!ring_take_warp(ring, kq++, abort_flag, p.status, w) || w < 0) break;
      const BUnit u = decode_bunit(p, w);
      if (!active) continue;
      bool ok = true;
      for (int i = 0; i < u.n_it && ok; ++i) {
        ok = mbar_wait_warp(dq_full, it_g & 1, abort_flag, p.status);
        if (!ok) break;
        tc_fence_after();
        uint32_t va[32], vb[32];
        tmem_ld32x2(tQ, tQ + 32, va, vb);
        tc_fence_before();
        mbar_arrive(dq_empty);  // these TMEM columns are free again
        const uint32_t k = kBoxes * it_g + 2 * rg;
        ok = stage_box(va, k) && stage_box(vb, k + 1);
        ++it_g;
      }
      if (!ok) break;
    }
  } else if (warp == 2 && !aborted_at_start) {
    // ------------------------------------------------------------ dQ reductions
    // Box kb (32 columns of one dQ tile) is issued as its own bulk group; once
    // box kb is in flight, box kb - 1 has had its source read when all groups
    // but the newest have, and its slot is handed back.
    if (lane == 0) {
      uint32_t kb = 0, kq = 0;
      bool ok = true;
      while (ok) {
        int w;
        if (!ring_take(ring, kq++, abort_flag, p.status, w) || w < 0) break;
        const BUnit u = decode_bunit(p, w);
        for (int i = 0; i < u.n_it && ok; ++i) {
          const int h = u.g * p.G + i / u.nq;
          const int qt = unit_qtile(u, i);
          const int plane = u.b * p.Hq + h;
          for (int j = 0; j < D / 32; ++j) {
            const uint32_t slot = kb & 1;
            ok = mbar_wait(stg_full + slot, (kb >> 1) & 1, abort_flag, p.status);
            if (!ok) break;
            tma_reduce_add_3d(&tmap_dq, smem + C::OFF_STG + slot * 16384, 32 * j, qt * kBM, plane);
            bulk_commit_group();
            if (kb >= 1) {
              bulk_wait_read_but1();
              const uint32_t kp = kb - 1;
              mbar_arrive(stg_read + 2 * (kp & 1) + ((kp % (D / 32)) >> 1));
            }
            ++kb;
          }
        }
      }
      bulk_wait_read_all();
      if (kb >= 1) {
        const uint32_t kp = kb - 1;
        mbar_arrive(stg_read + 2 * (kp & 1) + ((kp % (D / 32)) >> 1));
      }
      bulk_wait_all();  // the reductions finish before the CTA's memory goes
    }
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
  if (threadIdx.x == 0) {
    if (ring_retire(p.ctr, p.aborts, *abort_flag != 0) != 0 && p.acc_flags != nullptr)
      atomicAnd(p.acc_flags, ~kAccZeroed);
  }
}

template <int D, bool kDrop>
static cudaError_t launch_bwd_t(const CUtensorMap& tq, const CUtensorMap& tk,
                                const CUtensorMap& tv, const CUtensorMap& tdo,
                                const CUtensorMap& tdq,
                                const BwdParams& p,
                                const void* out, const void* out16, const float* lse,
                                const void* dout, void* dq, int stages,
                                int num_sms,
                                cudaStream_t stream, const BwdPrep* prep) {
  using C = BwdCfg<D>;
  static bool attr_set[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(bd_bwd_kernel<D, kDrop>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  const int planes = p.B * p.Hq;
  // out16 lacks the dropout scale that out carries
  const float o16_scale = kDrop ? p.drop.rp : 1.f;
  if ((stages & kBwdPrepare) && prep != nullptr) {
    cudaError_t e = launch_prep_bwd(*prep, out, out16, o16_scale, dout, lse, D, planes, p.L,
                                    p.Lq, const_cast<float*>(p.nlse2),
                                    const_cast<float*>(p.ndelta), p.dqacc, p.status, stream);
    if (e != cudaSuccess) return e;
  } else if (stages & kBwdPrepare) {
    const long long threads = (long long)planes * p.Lq * pre_threads_per_row<D>();
    bwd_pre_kernel<D><<<static_cast<unsigned>((threads + 255) / 256), 256, 0, stream>>>(
        static_cast<const __nv_bfloat16*>(out), static_cast<const __half*>(out16), o16_scale,
        static_cast<const __nv_bfloat16*>(dout), lse, planes, p.L, p.Lq,
        const_cast<float*>(p.nlse2), const_cast<float*>(p.ndelta), p.dqacc);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  const int grid = p.n_units < num_sms ? p.n_units : num_sms;
  if ((stages & kBwdMain) && grid > 0) {
    bd_bwd_kernel<D, kDrop><<<grid, kThreads, C::SMEM, stream>>>(tq, tk, tv, tdo, tdq, p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (stages & kBwdFinish) {
    const long long n8 = (long long)planes * p.L * D / 8;
    bwd_dq_kernel<D><<<static_cast<unsigned>((n8 + 255) / 256), 256, 0, stream>>>(
        p.dqacc, static_cast<__nv_bfloat16*>(dq), n8, p.scale);
  }
  return cudaGetLastError();
}

cudaError_t launch_bwd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const CUtensorMap& tdo, const CUtensorMap& tdq, const AttnDims& d,
                       void* plan, const void* out, const void* out16, const float* lse,
                       const void* dout, void* dq, void* dk,
                       void* dv, void* workspace, int32_t* status, int stages, int num_sms,
                       cudaStream_t stream, const BwdPrep* prep) {
  const PlanLayout pl = plan_layout(d.B, d.Hq, d.Hkv, d.L, d.S);
  const BwdLayout wl = bwd_layout(d.B, d.Hq, d.Hkv, d.L, d.S, d.D);
  char* base = static_cast<char*>(plan);
  char* ws = static_cast<char*>(workspace);
  BwdParams p{};
  p.B = d.B;
  p.Hq = d.Hq;
  p.Hkv = d.Hkv;
  p.L = d.L;
  p.S = d.S;
  p.seq_start = d.seq_start;
  p.G = d.Hq / d.Hkv;
  p.NKT = pl.NKT;
  p.Spad = pl.Spad;
  p.Lq = wl.Lq;
  p.n_units = d.B * pl.NKT * d.Hkv;
  p.scale_log2 = d.scale_log2;
  p.scale = d.scale;
  p.kend = reinterpret_cast<const int32_t*>(base + pl.kend);
  p.bwd_range = reinterpret_cast<const int32_t*>(base + pl.bwd_range);
  p.bwd_order = reinterpret_cast<const int32_t*>(base + pl.bwd_order);
  p.nlse2 = reinterpret_cast<const float*>(ws + wl.lsed);
  p.ndelta = p.nlse2 + (size_t)d.B * d.Hq * wl.Lq;
  p.dqacc = reinterpret_cast<float*>(ws + wl.dqacc);
  p.dk = static_cast<__nv_bfloat16*>(dk);
  p.dv = static_cast<__nv_bfloat16*>(dv);
  p.status = status;
  p.ctr = reinterpret_cast<int*>(base + pl.sched) + 2;
  p.aborts = reinterpret_cast<int*>(base + pl.sched) + 5;
  p.acc_flags = prep != nullptr ? &prep->hdr->flags : nullptr;
  p.wait_limit_ns = (stages & kBwdMain) ? take_wait_test(kWaitTestBwd, &p.withhold)
                                         : static_cast<uint32_t>(kWaitTimeoutNs);
  p.drop = d.drop;
  if (d.drop.on) {
    if (d.D == 64)
      return launch_bwd_t<64, true>(tq, tk, tv, tdo, tdq, p, out, out16, lse, dout, dq, stages,
                                    num_sms, stream, prep);
    return launch_bwd_t<128, true>(tq, tk, tv, tdo, tdq, p, out, out16, lse, dout, dq, stages,
                                   num_sms, stream, prep);
  }
  if (d.D == 64)
    return launch_bwd_t<64, false>(tq, tk, tv, tdo, tdq, p, out, out16, lse, dout, dq, stages,
                                   num_sms, stream, prep);
  return launch_bwd_t<128, false>(tq, tk, tv, tdo, tdq, p, out, out16, lse, dout, dq, stages,
                                  num_sms, stream, prep);
}

}  // namespace bd
