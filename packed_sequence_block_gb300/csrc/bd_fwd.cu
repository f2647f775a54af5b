// Forward pass of block-diagonal causal attention (cp_blockdiag_sdpa on the
// page "nemo_automodel.components.distributed.blockdiag_cp": local queries
// against the full key/value row under a per-document causal mask).
//
// Design (sm_103a):
//  * persistent CTAs (one per SM) walk a longest-first list of work units;
//    a unit is one query block = two 128-row sub-tiles that share every
//    key/value tile: two query heads of one GQA group (Hq/Hkv even) or two
//    consecutive row tiles of one head (Hq/Hkv odd);
//  * warp 0 streams Q and K/V tiles with TMA (128-byte swizzle) into shared
//    memory; only the key tiles the plan marks non-empty are loaded;
//  * warp 1 (one thread) issues tcgen05 MMAs: S_s = Q_s K^T into TMEM, then
//    O_s += P_s V with P_s read back from TMEM (fp16, with V read from the
//    fp16 copy that v_to_f16 writes before the kernel starts);
//  * warpgroups 1 and 2 run the softmax of sub-tile 0 and 1 (one thread per
//    query row = one TMEM lane): mask, running max, exp2, bf16 P into TMEM,
//    lazy rescaling of O, and the epilogue O / l -> bf16 plus the fp32 LSE.
// TMEM columns: S0 [0,128), S1 [128,256), O0 [256,256+D), O1 [384,384+D).
#include "bd_ptx.cuh"

namespace bd {

namespace {

constexpr int kThreads = 384;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale O when the max grows by > 2^8
constexpr float kLn2 = 0.6931471805599453f;

template <int D>
struct FwdCfg {
  static constexpr int QTILE = kBM * D * 2;  // bytes of one 128-row bf16 tile
  static constexpr int KTILE = kBN * D * 2;
  // A K stage frees once the S products of its tile are done, a V stage only
  // once the P V products are.  At D = 128 a third V stage measured no faster
  // than two, and its 32 KB stage the epilogue's stores instead.
  static constexpr int KSTAGES = (D == 64) ? 3 : 2;
  static constexpr int VSTAGES = (D == 64) ? 4 : 2;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + 2 * QTILE;
  static constexpr int OFF_V = OFF_K + KSTAGES * KTILE;
  // epilogue staging: per softmax warp 32 rows x 64 B of out, then of out16
  static constexpr int OFF_STG = OFF_V + VSTAGES * KTILE;
  static constexpr int OFF_BAR = OFF_STG + 8 * 4096;
  static constexpr int SMEM = OFF_BAR + 512;
  static constexpr uint32_t IDESC_S = make_idesc_bf16(128, 128, 0, 0);
  // P V runs with fp16 operands (V from its fp16 copy, P <= 2^8 by the
  // rescale threshold): O then carries P to 11 significant bits, and the
  // backward's Delta = <dO, O> agrees with its own P to that precision.
  static constexpr uint32_t IDESC_PV = make_idesc(128, D, 0, 1, 0);
};

struct FwdParams {
  int B, Hq, Hkv, L, S, seq_start, G, HP, NQB, Lpad, n_units, g_odd;
  float scale_log2;
  const int32_t* qlo;
  const int32_t* fwd_range;
  const int32_t* fwd_order;
  __nv_bfloat16* out;
  // optional: fp16 copy of O without the dropout scale 1 / (1 - p), i.e. the
  // normalised P V (within the range of v), from which the backward forms Delta
  __half* out16;
  float* lse;
  int32_t* status;
  int* ctr;  // work counters in the plan: [next unit, finished CTAs]
  int* aborts;  // CTAs of the launch that gave up a wait (in the plan)
  float4* acc;            // optional: zeroed by the idle warps (the backward's dq accumulator)
  long long acc_n16;      // its size in 16-byte words
  uint32_t* acc_flags;    // optional: gets kAccZeroed when every CTA finished cleanly
  uint32_t wait_limit_ns;  // bound of every device-side wait
  int withhold;            // test only: the producer withholds the first Q load
  DropoutArgs drop;
};

__device__ __forceinline__ void sts128(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                       uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}

// TMA store of a shared-memory box into global memory (rows past the
// tensor's extent are not written).
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, uint32_t smem_src, int c0,
                                             int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(smem_src), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

struct Unit {
  int b, h0, h1, qt0, qt1, kt_lo, n, g;
};

__device__ __forceinline__ Unit decode_unit(const FwdParams& p, int w) {
  const int per = p.Hkv * p.HP;
  const int e = w / per, r = w % per;
  const int qbl = p.fwd_order[e];
  Unit u;
  u.b = qbl / p.NQB;
  const int qb = qbl % p.NQB;
  u.g = r / p.HP;
  const int slot = r % p.HP;
  if (!p.g_odd) {
    u.h0 = u.g * p.G + 2 * slot;
    u.h1 = u.h0 + 1;
    u.qt0 = u.qt1 = qb;
  } else {
    u.h0 = u.h1 = u.g * p.G + slot;
    u.qt0 = 2 * qb;
    u.qt1 = 2 * qb + 1;
  }
  u.kt_lo = p.fwd_range[2 * qbl];
  u.n = p.fwd_range[2 * qbl + 1] - u.kt_lo + 1;
  return u;
}

// The decoded unit of each work-ring slot, written by the producer before it
// publishes the slot, so that the consumers read it from shared memory
// instead of repeating the dependent global loads of decode_unit.
struct UnitSlots {
  int4 a[kRing];  // b, h0, h1, qt0
  int4 b[kRing];  // qt1, kt_lo, n, g
};

// Producer: fetch this CTA's k-th unit, decode it into its slot and publish
// it (w = -1: no more work).
__device__ __forceinline__ bool publish_unit(WorkRing* r, UnitSlots* us, uint32_t k,
                                             const FwdParams& p, volatile int* abort, int& w,
                                             Unit& u) {
  const int slot = k % kRing;
  if (!mbar_wait(&r->empty[slot], ((k / kRing) & 1) ^ 1, abort, p.status)) return false;
  w = atomicAdd(&p.ctr[0], 1);
  if (w >= p.n_units) w = -1;
  if (w >= 0) {
    u = decode_unit(p, w);
    // plain stores: the arrive below (an asm statement with a memory clobber)
    // keeps them before it, and it releases them to the slot's consumers
    us->a[slot] = make_int4(u.b, u.h0, u.h1, u.qt0);
    us->b[slot] = make_int4(u.qt1, u.kt_lo, u.n, u.g);
  }
  *reinterpret_cast<volatile int*>(&r->idx[slot]) = w;
  mbar_arrive(&r->full[slot]);
  return true;
}

__device__ __forceinline__ Unit slot_unit(const UnitSlots* us, int slot) {
  const int4 a = us->a[slot];  // after the slot's full wait (acquire)
  const int4 b = us->b[slot];
  Unit u;
  u.b = a.x; u.h0 = a.y; u.h1 = a.z; u.qt0 = a.w;
  u.qt1 = b.x; u.kt_lo = b.y; u.n = b.z; u.g = b.w;
  return u;
}

// Consumers: take slot k's unit (one thread, or a whole warp whose lane 0
// releases the slot).
__device__ __forceinline__ bool take_unit(WorkRing* r, const UnitSlots* us, uint32_t k,
                                          volatile int* abort, int32_t* status, int& w, Unit& u) {
  const int slot = k % kRing;
  if (!mbar_wait(&r->full[slot], (k / kRing) & 1, abort, status)) return false;
  w = *reinterpret_cast<volatile int*>(&r->idx[slot]);
  if (w >= 0) u = slot_unit(us, slot);
  mbar_arrive(&r->empty[slot]);
  return true;
}
__device__ __forceinline__ bool take_release_unit_warp(WorkRing* r, const UnitSlots* us,
                                                       uint32_t k, volatile int* abort,
                                                       int32_t* status, int& w, Unit& u) {
  const int slot = k % kRing;
  if (!mbar_wait_warp(&r->full[slot], (k / kRing) & 1, abort, status)) return false;
  w = *reinterpret_cast<volatile int*>(&r->idx[slot]);
  if (w >= 0) u = slot_unit(us, slot);
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(&r->empty[slot]);
  return true;
}
// A second warp form leaves the slot taken: the warp reads the unit again
// when it starts it (holding no registers meanwhile) and then releases it.
__device__ __forceinline__ bool take_unit_warp(WorkRing* r, uint32_t k, volatile int* abort,
                                               int32_t* status, int& w) {
  const int slot = k % kRing;
  if (!mbar_wait_warp(&r->full[slot], (k / kRing) & 1, abort, status)) return false;
  w = *reinterpret_cast<volatile int*>(&r->idx[slot]);
  return true;
}
__device__ __forceinline__ Unit release_unit_warp(WorkRing* r, const UnitSlots* us, uint32_t k) {
  const int slot = k % kRing;
  const Unit u = slot_unit(us, slot);
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(&r->empty[slot]);
  return u;
}

// Bounded wait used at teardown for copies/MMAs already in flight: ignores
// the abort flag (the operation completes on its own) but never spins forever.
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity, int32_t* status) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > kWaitTimeoutNs) {
      set_status(status, BD_ERR_TIMEOUT);
      return;
    }
  }
}

}  // namespace

// kDrop: attention dropout on the weights that feed P V (p.drop): a dropped
// weight is written as 0 into the P tile and the kept ones are scaled by
// 1 / (1 - p) with 1 / l in the epilogue; the row sum and the log-sum-exp stay
// those of the undropped softmax.
template <int D, bool kDrop>
__global__ void __launch_bounds__(kThreads, 1)
    bd_fwd_kernel(const __grid_constant__ CUtensorMap tmap_q,
                  const __grid_constant__ CUtensorMap tmap_k,
                  const __grid_constant__ CUtensorMap tmap_v,
                  const __grid_constant__ CUtensorMap tmap_o,
                  const __grid_constant__ CUtensorMap tmap_o16,
                  const __grid_constant__ FwdParams p) {
  using C = FwdCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* q_full = bars + 0;
  uint64_t* q_empty = bars + 1;
  uint64_t* k_full = bars + 2;                      // [KSTAGES]
  uint64_t* k_empty = k_full + C::KSTAGES;          // [KSTAGES]
  uint64_t* v_full = k_empty + C::KSTAGES;          // [VSTAGES]
  uint64_t* v_empty = v_full + C::VSTAGES;          // [VSTAGES]
  uint64_t* s_full = v_empty + C::VSTAGES;          // [2]
  uint64_t* p_full = s_full + 2;                    // [2]
  uint64_t* o_full = p_full + 2;                    // [2]
  uint64_t* drain = o_full + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);  // + the wait limit
  WorkRing* ring = reinterpret_cast<WorkRing*>(smem + C::OFF_BAR + 256);
  UnitSlots* uslots = reinterpret_cast<UnitSlots*>(smem + C::OFF_BAR + 384);
  static_assert(256 + sizeof(WorkRing) <= 384, "ring past the unit slots");
  static_assert(384 + sizeof(UnitSlots) <= C::SMEM - C::OFF_BAR, "barrier area too small");
  static_assert(C::SMEM <= 232448, "shared memory over the per-block limit");

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    abort_flag[0] = 0;
    abort_flag[1] = static_cast<int>(p.wait_limit_ns);
    if ((smem_u32(smem) & 1023u) != 0) {  // swizzled tiles need 1024-byte alignment
      set_status(p.status, BD_ERR_CUDA);
      *abort_flag = 1;
    }
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    for (int s = 0; s < C::KSTAGES; ++s) {
      mbar_init(k_full + s, 1);
      mbar_init(k_empty + s, 1);
    }
    for (int s = 0; s < C::VSTAGES; ++s) {
      mbar_init(v_full + s, 1);
      mbar_init(v_empty + s, 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(s_full + s, 1);
      mbar_init(p_full + s, 128);
      mbar_init(o_full + s, 1);
    }
    mbar_init(drain, 1);
    ring_init(ring, 9);  // MMA thread + 8 softmax warps
    fence_mbar_init();
    prefetch_tmap(&tmap_q);
    prefetch_tmap(&tmap_k);
    prefetch_tmap(&tmap_v);
    prefetch_tmap(&tmap_o);
    prefetch_tmap(&tmap_o16);
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
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t k_it = 0, v_it = 0, u_it = 0, kq = 0;
      bool q_issued = false;
      for (;;) {
        int w;
        Unit u;
        if (!publish_unit(ring, uslots, kq++, p, abort_flag, w, u) || w < 0) break;
        if (u.n <= 0) continue;
        // test of the bounded waits: the unit is published but its Q never
        // arrives, so the MMA thread's wait for it runs out
        if (p.withhold) break;
        if (!mbar_wait(q_empty, (u_it & 1) ^ 1, abort_flag, p.status)) break;
        mbar_arrive_expect_tx(q_full, 2 * C::QTILE);
        q_issued = true;
        for (int j = 0; j < D / 64; ++j) {
          tma_load_3d(smem + C::OFF_Q + j * 16384, &tmap_q, q_full, 64 * j, u.qt0 * kBM,
                      u.b * p.Hq + u.h0);
          tma_load_3d(smem + C::OFF_Q + C::QTILE + j * 16384, &tmap_q, q_full, 64 * j,
                      u.qt1 * kBM, u.b * p.Hq + u.h1);
        }
        ++u_it;
        const int plane = u.b * p.Hkv + u.g;
        bool ok = true;
        for (int jj = 0; jj < u.n; ++jj) {
          const int row = (u.kt_lo + jj) * kBN;
          const int st = k_it % C::KSTAGES;
          ok = mbar_wait(k_empty + st, ((k_it / C::KSTAGES) & 1) ^ 1, abort_flag, p.status);
          if (!ok) break;
          mbar_arrive_expect_tx(k_full + st, C::KTILE);
          for (int j = 0; j < D / 64; ++j)
            tma_load_3d(smem + C::OFF_K + st * C::KTILE + j * 16384, &tmap_k, k_full + st, 64 * j,
                        row, plane);
          ++k_it;
          const int sv = v_it % C::VSTAGES;
          ok = mbar_wait(v_empty + sv, ((v_it / C::VSTAGES) & 1) ^ 1, abort_flag, p.status);
          if (!ok) break;
          mbar_arrive_expect_tx(v_full + sv, C::KTILE);
          for (int j = 0; j < D / 64; ++j)
            tma_load_3d(smem + C::OFF_V + sv * C::KTILE + j * 16384, &tmap_v, v_full + sv, 64 * j,
                        row, plane);
          ++v_it;
        }
        if (!ok) break;
      }
      // teardown: every issued copy must land before the CTA's memory is released
      if (q_issued) drain_wait(q_full, (u_it - 1) & 1, p.status);
      for (int st = 0; st < C::KSTAGES; ++st) {
        if (k_it > static_cast<uint32_t>(st)) {
          const uint32_t last = k_it - 1 - ((k_it - 1 - st) % C::KSTAGES);
          drain_wait(k_full + st, (last / C::KSTAGES) & 1, p.status);
        }
      }
      for (int st = 0; st < C::VSTAGES; ++st) {
        if (v_it > static_cast<uint32_t>(st)) {
          const uint32_t last = v_it - 1 - ((v_it - 1 - st) % C::VSTAGES);
          drain_wait(v_full + st, (last / C::VSTAGES) & 1, p.status);
        }
      }
    }
    __syncwarp();
  } else if (warp == 1 && !aborted_at_start) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t sq0 = smem_u32(smem + C::OFF_Q);
      const uint32_t sk0 = smem_u32(smem + C::OFF_K);
      const uint32_t sv0 = smem_u32(smem + C::OFF_V);
      // each operand's descriptor is built once per product and stepped by
      // a constant per instruction (sdesc_add), keeping this thread's
      // instruction count per tcgen05.mma low
      auto issue_s = [&](int s, int st) {
        const uint64_t qd = make_sdesc_sw128(sq0 + s * C::QTILE, 16, 1024);
        const uint64_t kd = make_sdesc_sw128(sk0 + st * C::KTILE, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
          if (kk == 0)
            mma_ss(tmem + s * 128, qd, kd, C::IDESC_S, 0);
          else
            mma_ss_acc(tmem + s * 128, sdesc_add(qd, off), sdesc_add(kd, off), C::IDESC_S);
        }
      };
      auto issue_pv = [&](int s, int st, bool acc) {
        const uint64_t vd = make_sdesc_sw128(sv0 + st * C::KTILE, 16384, 1024);
#pragma unroll
        for (int ks = 0; ks < kBN / 16; ++ks) {
          if (ks == 0)
            mma_ts(tmem + 256 + s * 128, tmem + s * 128, vd, C::IDESC_PV, acc);
          else
            mma_ts_acc(tmem + 256 + s * 128, tmem + s * 128 + ks * 8, sdesc_add(vd, ks * 2048),
                       C::IDESC_PV);
        }
      };
      uint32_t kv_it = 0, u_it = 0, t_it = 0, kq = 0;
      bool ok = true;
      while (ok) {
        int w;
        Unit u;
        if (!take_unit(ring, uslots, kq++, abort_flag, p.status, w, u) || w < 0) break;
        if (u.n <= 0) continue;
        ok = mbar_wait(q_full, u_it & 1, abort_flag, p.status);
        if (!ok) break;
        int st = kv_it % C::KSTAGES;
        ok = mbar_wait(k_full + st, (kv_it / C::KSTAGES) & 1, abort_flag, p.status);
        if (!ok) break;
        tc_fence_after();
        issue_s(0, st);
        mma_commit(s_full + 0);
        issue_s(1, st);
        mma_commit(s_full + 1);
        // only the S products read Q: once the unit's last ones are issued the
        // producer may load the next unit's Q behind them
        if (u.n == 1) mma_commit(q_empty);
        for (int jj = 0; jj < u.n && ok; ++jj) {
          const uint32_t it = kv_it + jj;
          const int stj = it % C::KSTAGES, svj = it % C::VSTAGES;
          mma_commit(k_empty + stj);  // the S MMAs reading K_jj are all issued
          ok = mbar_wait(v_full + svj, (it / C::VSTAGES) & 1, abort_flag, p.status);
          if (!ok) break;
          const bool last = (jj + 1 == u.n);
          const int stn = (it + 1) % C::KSTAGES;
          for (int s = 0; s < 2 && ok; ++s) {
            ok = mbar_wait(p_full + s, t_it & 1, abort_flag, p.status);
            if (!ok) break;
            tc_fence_after();
            issue_pv(s, svj, jj > 0);
            if (!last) {
              if (s == 0) {
                ok = mbar_wait(k_full + stn, ((it + 1) / C::KSTAGES) & 1, abort_flag, p.status);
                if (!ok) break;
                tc_fence_after();
              }
              issue_s(s, stn);
              mma_commit(s_full + s);
              if (s == 1 && jj + 2 == u.n) mma_commit(q_empty);
            } else {
              mma_commit(o_full + s);
            }
          }
          mma_commit(v_empty + svj);
          ++t_it;
        }
        kv_it += u.n;
        ++u_it;
      }
      // teardown: wait for every MMA issued so far
      mma_commit(drain);
      drain_wait(drain, 0, p.status);
    }
    __syncwarp();
  } else if (warp >= 4 && !aborted_at_start) {
    // ------------------------------------------------------------ softmax
    const int wg = (warp - 4) >> 2;  // sub-tile
    const int q4 = warp & 3;
    const int r = q4 * 32 + lane;     // row of the sub-tile = TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(q4 * 32) << 16;
    const uint32_t tS = tmem + lane_off + wg * 128;
    const uint32_t tO = tmem + lane_off + 256 + wg * 128;
    uint32_t t_it = 0, o_it = 0, kq = 0;
    // The next unit is taken from the ring ahead of time (at the current
    // unit's epilogue, when the producer has published it: it only waits for
    // stages that this unit's P tiles have already released), and the load of
    // this row's mask bound is issued then, so that neither lies between one
    // unit's epilogue and the next unit's first tile (~2,900 cycles a unit
    // when they did).
    // At D = 128 the slot stays taken until the unit starts (no registers
    // held across the epilogue); at D = 64 the unit is read and the slot
    // released at once (the other form measured 2.6% slower there).
    int nw = -1;
    Unit nu{};
    int32_t nlo = kPadLo;
    auto take_next = [&]() -> bool {
      if constexpr (D == 128) {
        if (!take_unit_warp(ring, kq, abort_flag, p.status, nw)) return false;
        if (nw >= 0) {
          const int4 a = uslots->a[kq % kRing], b = uslots->b[kq % kRing];  // b,..,..,qt0 | qt1
          const int ni = (wg ? b.x : a.w) * kBM + r;
          nlo = ni < p.L ? p.qlo[(size_t)a.x * p.Lpad + ni] : kPadLo;
        } else {
          release_unit_warp(ring, uslots, kq);
        }
        ++kq;
      } else {
        if (!take_release_unit_warp(ring, uslots, kq++, abort_flag, p.status, nw, nu)) return false;
        if (nw >= 0) {
          const int ni = (wg ? nu.qt1 : nu.qt0) * kBM + r;
          nlo = ni < p.L ? p.qlo[(size_t)nu.b * p.Lpad + ni] : kPadLo;
        }
      }
      return true;
    };
    bool have = take_next();
    while (have && nw >= 0) {
      Unit u = nu;
      if constexpr (D == 128) u = release_unit_warp(ring, uslots, kq - 1);
      const int h = wg ? u.h1 : u.h0;
      const int qt = wg ? u.qt1 : u.qt0;
      const int i = qt * kBM + r;  // local query row
      const bool in_range = i < p.L;
      const int t = p.seq_start + i;
      const uint32_t tpos = static_cast<uint32_t>(t);  // dropout counter word 1
      const uint32_t plane = static_cast<uint32_t>(u.b * p.Hq + h);
      const int32_t lo = nlo;
      const size_t row = static_cast<size_t>(u.b * p.Hq + h) * p.L + i;
      if (u.n <= 0) {
        if (in_range) {
          uint4* dst = reinterpret_cast<uint4*>(p.out + row * D);
#pragma unroll
          for (int c = 0; c < D / 8; ++c) dst[c] = make_uint4(0, 0, 0, 0);
          if (p.out16 != nullptr) {
            uint4* dl = reinterpret_cast<uint4*>(p.out16 + row * D);
#pragma unroll
            for (int c = 0; c < D / 8; ++c) dl[c] = make_uint4(0, 0, 0, 0);
          }
          p.lse[row] = -INFINITY;
        }
        have = take_next();
        continue;
      }
      float m_used = -INFINITY, l = 0.f;
      bool ok = true;
      for (int jj = 0; jj < u.n; ++jj) {
        const int k0 = (u.kt_lo + jj) * kBN;
        ok = mbar_wait_warp(s_full + wg, t_it & 1, abort_flag, p.status);
        if (!ok) break;
        tc_fence_after();
        // allowed columns of this tile for this row: [ca, cb]
        int ca = 1, cb = 0;
        if (lo != kPadLo) {
          ca = lo - k0;
          cb = t - k0;
        }
        const bool full = __all_sync(0xffffffffu, ca <= 0 && cb >= kBN - 1);
        // the row's 128 scores in one read; masked ones become -inf, which
        // neither raises the max nor adds to the sum (exp2(-inf) = 0)
        uint32_t v[128];
        tmem_ld128(tS, v);
        if (!full) {
          uint32_t mw[4];  // allowed columns [ca, cb], 32 per word
#pragma unroll
          for (int w = 0; w < 4; ++w) {
            const int lo = max(ca - 32 * w, 0), hi = min(cb - 32 * w, 31);
            mw[w] = (lo > hi) ? 0u
                              : ((0xffffffffu >> (31 - max(hi, 0))) & (0xffffffffu << min(lo, 31)));
          }
#pragma unroll
          for (int e = 0; e < kBN; ++e)
            v[e] = ((mw[e >> 5] >> (e & 31)) & 1u) ? v[e] : 0xff800000u;
        }
        // row max over four independent chains of three-input maxima
        float m4[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) m4[j] = fmaxf(__uint_as_float(v[j]), __uint_as_float(v[j + 4]));
#pragma unroll
        for (int e = 8; e < kBN; e += 8) {
#pragma unroll
          for (int j = 0; j < 4; ++j)
            m4[j] = fmax3(m4[j], __uint_as_float(v[e + j]), __uint_as_float(v[e + 4 + j]));
        }
        const float mx = fmax3(fmaxf(m4[0], m4[1]), m4[2], m4[3]);
        const float m_tile = mx * p.scale_log2;
        const float m_new = fmaxf(m_used, m_tile);
        float factor = 1.f;
        bool rescale = false;
        if (m_new != -INFINITY) {
          if (m_used == -INFINITY) {
            m_used = m_new;  // nothing accumulated yet for this row (O row is 0)
          } else if (m_new > m_used + kRescaleThreshold) {
            factor = fast_exp2(m_used - m_new);
            l *= factor;
            m_used = m_new;
            rescale = true;
          }
        }
        // P = exp2(s * scale * log2 e - m) as fp16 pairs into the S columns; the
        // row sum over eight independent partial sums
        const float m_use = (m_used == -INFINITY) ? 0.f : m_used;
        const float2 sc2 = make_float2(p.scale_log2, p.scale_log2), nm2 = make_float2(-m_use, -m_use);
        float2 l4[4];  // eight partial sums, as pairs
#pragma unroll
        for (int j = 0; j < 4; ++j) l4[j] = make_float2(0.f, 0.f);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t pk[16];
          uint4 w = make_uint4(0, 0, 0, 0);  // Philox words of the current eight keys
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            const float2 t = ffma2(make_float2(__uint_as_float(v[c * 32 + e]),
                                               __uint_as_float(v[c * 32 + e + 1])), sc2, nm2);
            const float2 x = make_float2(fast_exp2(t.x), fast_exp2(t.y));
            l4[(e >> 1) & 3] = fadd2(l4[(e >> 1) & 3], x);
            if constexpr (kDrop) {
              // key j = k0 + c*32 + e: counter (j >> 3, t, plane, offset); keys e and
              // e + 1 take the low and high halves of word (j & 7) >> 1
              if ((e & 7) == 0)
                w = philox4x32_10(static_cast<uint32_t>((k0 + c * 32 + e) >> 3), tpos, plane,
                                  p.drop.offset, p.drop.rk);
              const uint32_t wd = (e & 7) == 0 ? w.x : (e & 7) == 2 ? w.y : (e & 7) == 4 ? w.z : w.w;
              pk[e >> 1] = pack_f16x2((wd & 0xffffu) >= p.drop.threshold ? x.x : 0.f,
                                      (wd >> 16) >= p.drop.threshold ? x.y : 0.f);
            } else {
              pk[e >> 1] = pack_f16x2(x.x, x.y);
            }
          }
          tmem_st16(tS + c * 16, pk);
        }
        l += ((l4[0].x + l4[0].y) + (l4[1].x + l4[1].y)) + ((l4[2].x + l4[2].y) + (l4[3].x + l4[3].y));
        if (__any_sync(0xffffffffu, rescale)) {
          // O holds P_0..P_{jj-1} times V (the S_full wait covered those MMAs);
          // done after P is written, when the scores no longer hold registers
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t ov[32];
            tmem_ld32(tO + c * 32, ov);
            uint32_t a[16], b2[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              a[e] = __float_as_uint(__uint_as_float(ov[e]) * factor);
              b2[e] = __float_as_uint(__uint_as_float(ov[16 + e]) * factor);
            }
            tmem_st16(tO + c * 32, a);
            tmem_st16(tO + c * 32 + 16, b2);
          }
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(p_full + wg);
        ++t_it;
      }
      if (!ok) break;
      // epilogue: O / l -> bf16, LSE (the next unit taken first)
      have = take_next();
      if (!have) break;
      ok = mbar_wait_warp(o_full + wg, o_it & 1, abort_flag, p.status);
      if (!ok) break;
      ++o_it;
      tc_fence_after();
      // the kept weights enter P V unscaled; 1 / (1 - p) joins 1 / l for out
      // (out16 keeps the normalised P V, whose entries lie within v's range)
      // LSE before the O chunks at D = 128 (m_used and l then leave the
      // registers before the row's 128 O values arrive); after them at D = 64
      if (D == 128 && in_range) p.lse[row] = (l > 0.f) ? (m_used + log2f(l)) * kLn2 : -INFINITY;
      const float inv16 = (l > 0.f) ? 1.f / l : 0.f;
      const float inv = kDrop ? inv16 * p.drop.rp : inv16;
      // Each 32-column chunk of this warp's 32 rows goes through its staging
      // area in the TMA box layout (64-byte rows, 16-byte pieces swizzled by
      // row pair, which also keeps the writes free of bank conflicts), and
      // lane 0 hands it to the TMA unit as one store per output: the global
      // writes then leave the warp's path.  The area is reused once the TMA has
      // read the previous chunk.
      const uint32_t stg = smem_u32(smem + C::OFF_STG) + (warp - 4) * 4096;
      const int i0 = i - lane;  // the warp's first row
      const int plane_o = u.b * p.Hq + h;
      // the row's D columns in one TMEM read (the scores no longer hold
      // registers), instead of one dependent read per chunk
      uint32_t ov[D];
      if constexpr (D == 128) {
        tmem_ld128(tO, ov);
      } else {
        uint32_t (&o0)[32] = *reinterpret_cast<uint32_t(*)[32]>(&ov[0]);
        uint32_t (&o1)[32] = *reinterpret_cast<uint32_t(*)[32]>(&ov[32]);
        tmem_ld32x2(tO, tO + 32, o0, o1);
      }
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        const uint32_t* v = ov + c * 32;
        uint32_t pk[16], pl[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const float a = __uint_as_float(v[2 * e]), b = __uint_as_float(v[2 * e + 1]);
          pk[e] = pack_bf16x2(a * inv, b * inv);
          pl[e] = pack_f16x2(a * inv16, b * inv16);
        }
        if (lane == 0) bulk_wait_read_all();  // the TMA has read the previous chunk
        __syncwarp();
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint32_t a = stg + lane * 64 + ((j ^ ((lane >> 1) & 3)) << 4);
          sts128(a, pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
          sts128(a + 2048, pl[4 * j], pl[4 * j + 1], pl[4 * j + 2], pl[4 * j + 3]);
        }
        fence_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_3d(&tmap_o, stg, c * 32, i0, plane_o);
          if (p.out16 != nullptr) tma_store_3d(&tmap_o16, stg + 2048, c * 32, i0, plane_o);
          bulk_commit_group();
        }
      }
      if (D == 64 && in_range) p.lse[row] = (l > 0.f) ? (m_used + log2f(l)) * kLn2 : -INFINITY;
      tc_fence_before();
    }
    if (lane == 0) bulk_wait_all();  // this warp's output stores are done
    __syncwarp();
  } else if ((warp == 2 || warp == 3) && p.acc != nullptr) {
    // ------------------------------------------------------------ zeroing
    // The two warps without a role zero the backward's dq accumulator while
    // the others compute, so that the backward need not make that pass.
    const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
    for (long long i = (long long)blockIdx.x * 64 + (warp - 2) * 32 + lane; i < p.acc_n16;
         i += (long long)gridDim.x * 64)
      p.acc[i] = z;
    __threadfence();
  }

  // ------------------------------------------------------------ teardown
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
  if (threadIdx.x == 0) {
    // the last CTA records the zeroed accumulator when no CTA gave up (one
    // that aborted at start skipped its share of the zeroing)
    if (ring_retire(p.ctr, p.aborts, *abort_flag != 0) == 1 && p.acc_flags != nullptr)
      atomicOr(p.acc_flags, kAccZeroed);
  }
}

template <int D, bool kDrop>
static cudaError_t launch_fwd_t(const CUtensorMap& tq, const CUtensorMap& tk,
                                const CUtensorMap& tv, const CUtensorMap& to,
                                const CUtensorMap& to16, const FwdParams& p, int num_sms,
                                cudaStream_t stream) {
  using C = FwdCfg<D>;
  static bool attr_set[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(bd_fwd_kernel<D, kDrop>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  const int grid = p.n_units < num_sms ? p.n_units : num_sms;
  if (grid <= 0) return cudaSuccess;
  bd_fwd_kernel<D, kDrop><<<grid, kThreads, C::SMEM, stream>>>(tq, tk, tv, to, to16, p);
  return cudaGetLastError();
}

// v (bf16) -> fp16, eight elements a thread per step of a grid-stride loop.
__global__ void __launch_bounds__(256) v_to_f16_kernel(const uint4* __restrict__ v,
                                                       uint4* __restrict__ v16, long long n8) {
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n8;
       i += (long long)gridDim.x * blockDim.x) {
    const uint4 x = v[i];
    v16[i] = make_uint4(bf16x2_to_f16x2(x.x), bf16x2_to_f16x2(x.y), bf16x2_to_f16x2(x.z),
                        bf16x2_to_f16x2(x.w));
  }
}

cudaError_t launch_v_to_f16(const void* v, void* v16, long long n, int num_sms,
                            cudaStream_t stream) {
  const long long n8 = n / 8;
  const long long want = (n8 + 255) / 256;
  const int blocks = static_cast<int>(want < 16LL * num_sms ? want : 16LL * num_sms);
  if (blocks <= 0) return cudaSuccess;
  v_to_f16_kernel<<<blocks, 256, 0, stream>>>(static_cast<const uint4*>(v),
                                              static_cast<uint4*>(v16), n8);
  return cudaGetLastError();
}

cudaError_t launch_fwd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const CUtensorMap& to, const CUtensorMap& to16, const AttnDims& d,
                       void* plan, void* out, void* out16, float* lse, int32_t* status,
                       int num_sms, cudaStream_t stream, void* acc, size_t acc_bytes,
                       uint32_t* acc_flags) {
  const PlanLayout pl = plan_layout(d.B, d.Hq, d.Hkv, d.L, d.S);
  char* base = static_cast<char*>(plan);
  FwdParams p{};
  p.B = d.B;
  p.Hq = d.Hq;
  p.Hkv = d.Hkv;
  p.L = d.L;
  p.S = d.S;
  p.seq_start = d.seq_start;
  p.G = d.Hq / d.Hkv;
  p.g_odd = p.G % 2;
  p.HP = p.g_odd ? p.G : p.G / 2;
  p.NQB = pl.NQB;
  p.Lpad = pl.Lpad;
  p.n_units = d.B * pl.NQB * d.Hkv * p.HP;
  p.scale_log2 = d.scale_log2;
  p.qlo = reinterpret_cast<const int32_t*>(base + pl.qlo);
  p.fwd_range = reinterpret_cast<const int32_t*>(base + pl.fwd_range);
  p.fwd_order = reinterpret_cast<const int32_t*>(base + pl.fwd_order);
  p.out = static_cast<__nv_bfloat16*>(out);
  p.out16 = static_cast<__half*>(out16);
  p.lse = lse;
  p.status = status;
  p.ctr = reinterpret_cast<int*>(base + pl.sched);
  p.aborts = p.ctr + 4;
  p.acc = static_cast<float4*>(acc);
  p.acc_n16 = static_cast<long long>(acc_bytes / 16);
  p.acc_flags = acc != nullptr ? acc_flags : nullptr;
  p.wait_limit_ns = take_wait_test(kWaitTestFwd, &p.withhold);
  p.drop = d.drop;
  if (d.drop.on) {
    if (d.D == 64) return launch_fwd_t<64, true>(tq, tk, tv, to, to16, p, num_sms, stream);
    return launch_fwd_t<128, true>(tq, tk, tv, to, to16, p, num_sms, stream);
  }
  if (d.D == 64) return launch_fwd_t<64, false>(tq, tk, tv, to, to16, p, num_sms, stream);
  return launch_fwd_t<128, false>(tq, tk, tv, to, to16, p, num_sms, stream);
}

}  // namespace bd
