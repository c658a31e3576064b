// Backward, dK/dV kernel for D = 256: each CTA owns a tile of BK = 128 key
// rows of one (batch, KV head) and loops over the G query heads of its group,
// then over the visible query tiles ("feat(attention): complete Flash
// Attention VJP implementation", section "Two-Kernel Design": grid [NK, kvH,
// B], loop over the GQA group then the Q blocks, K-row ownership so dK and dV
// need no atomics).  Per query tile everything is computed transposed, so the
// key row is the TMEM lane:
//   S^T = K Q^T, dP^T = V dO^T                       (tcgen05, fp32 in TMEM)
//   P^T = exp2(S^T * scale_log2 - lse), dS^T = P^T * (dP^T - delta)
//   dV += P^T dO, dK += dS^T Q                        (tcgen05, A from TMEM)
// and finally dK is scaled by `scale`.
//
// At D = 256 the dK and dV accumulators alone fill the 512 TMEM columns, so
// the two CTAs of a cluster share a key tile (attn_bwd_dkv_kernel below):
// the dV CTA computes S^T, P^T and dV and hands P^T (16-bit, the values its
// own dV MMA uses) to the dK CTA through distributed shared memory; the dK
// CTA computes dP^T, forms dS^T from the received P^T and accumulates dK.
// Each CTA issues two of the four products per query tile, and S^T is
// computed once.  P^T and dS^T (16-bit pairs) are written over fp32 columns
// the row threads have just read, and the MMA that next writes those columns
// is issued after the MMAs that read them by the same thread (tcgen05 MMAs of
// one thread run in issue order).
//
// Warp roles (320 threads): warps 0-7 row threads -- warp w owns TMEM lanes
// 32*(w%4)..+31 (key rows) and query columns 32*(w/4)..+31 of each tile;
// warp 8 producer (TMA for Q/dO tiles, plain loads for the per-query
// lse/delta values); warp 9 MMA issuer and TMEM owner.
#pragma once

#include "kernel_common.cuh"

namespace gbattn {

// P^T of one query tile handed from the dV CTA to the dK CTA of a cluster:
// 128 key rows x 64 queries of 16-bit values, 128 bytes per row as eight
// 16-byte chunks (chunk j holds queries 8j..8j+7), chunk j of row r stored at
// position j ^ (r & 7) so that the 32 rows of a warp spread over all banks.
// Two slots: the dV CTA may run one query tile ahead.
struct PtXch {
  static constexpr int SLOT_BYTES = 128 * 128;
  static constexpr int SLOTS = 2;
  static constexpr int BYTES = SLOTS * SLOT_BYTES;
  __device__ __forceinline__ static uint32_t addr(uint32_t base, int slot, int r, int chunk) {
    return base + slot * SLOT_BYTES + r * 128 + ((chunk ^ (r & 7)) << 4);
  }
};

// mbarriers of the hand-off, in the shared memory of both CTAs (the kernel
// declares them, so they sit at the same offset in either CTA).  pfull, in
// the dK CTA: one local arrival that expects the slot's bytes, which the dV
// CTA's asynchronous stores complete (the bytes are visible to a thread that
// sees the phase complete, as for a TMA load).  pfree, in the dV CTA: one
// arrival per warp of the dK CTA's row threads once they have used the
// slot's values.
struct PtXchBars {
  uint64_t pfull[PtXch::SLOTS], pfree[PtXch::SLOTS];
};

// D = 256, dK half (cluster rank 1).  V sits in tensor memory as the A
// operand of dP^T = V dO^T (copied in by the row threads), so only the
// dO^T tile is read from shared memory; P^T comes from the partner CTA.
// Tensor memory: dK (256 columns), V (128: 256 16-bit values per row), dP^T
// (two buffers of 64).  The row threads write dS^T (16-bit pairs) over the
// dP^T columns they have read, and the MMA warp issues dK += dS^T Q, then
// dP^T of the tile after next into the same buffer (tcgen05 MMAs of one
// thread run in issue order).
struct Dk256Geom {
  static constexpr int D = 256, BK = 128, BQ = 64, NCH = 4;
  static constexpr int Q_BYTES = NCH * BQ * 128;  // 32 KB
  static constexpr int STATIC_EST = 2048;         // static shared memory of the pair kernel, upper estimate
  static constexpr int STAGES_FIT = (kMaxDynSmem - STATIC_EST - 1024 - PtXch::BYTES) / (2 * Q_BYTES);
  static constexpr int STAGES = STAGES_FIT > 3 ? 3 : STAGES_FIT;
  static constexpr int XCH_OFF = STAGES * 2 * Q_BYTES;  // from the 1024-aligned base
  static constexpr int SMEM_BYTES = 1024 + XCH_OFF + PtXch::BYTES;
  static constexpr int DK_COL = 0, V_COL = 256, DPT_COL = 384;  // dP^T: 2 x 64
  static constexpr int TMEM_COLS = 512;
  static constexpr int NUM_COMPUTE_WARPS = 8;
  static constexpr int NCT = 32 * NUM_COMPUTE_WARPS;
  static constexpr int PRODUCER_WARP = NUM_COMPUTE_WARPS;
  static constexpr int MMA_WARP = NUM_COMPUTE_WARPS + 1;
  static constexpr int NUM_THREADS = 32 * (NUM_COMPUTE_WARPS + 2);
  static_assert(STAGES >= 3, "three Q/dO stages: dP^T runs two query tiles ahead");
  static_assert(DPT_COL + 2 * BQ <= TMEM_COLS, "tensor memory budget");
};

template <bool BF16, bool CAUSAL, bool MASKED>
__device__ __forceinline__ void dk256_tile(const CUtensorMap& tmQ, const CUtensorMap& tmdO, const BwdParams& p,
                                           const int bhk, const int kt, PtXchBars& xb) {
  using Gm = Dk256Geom;
  using E = Elem<BF16>;
  constexpr int D = Gm::D, BQ = Gm::BQ, BK = Gm::BK, NCH = Gm::NCH, ST = Gm::STAGES, NCT = Gm::NCT;

  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t bar_vready, bar_stfull[ST], bar_stempty[ST], bar_dpfull[2], bar_dsready[2], bar_accdone;
  __shared__ __align__(16) float dlt_s[ST][BQ];
  __shared__ uint32_t tmem_slot;
  __shared__ volatile int abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t sQ0 = sbase;
  const uint32_t sdO0 = sQ0 + ST * Gm::Q_BYTES;
  const uint32_t sX = sbase + Gm::XCH_OFF;

  const int b = bhk / p.Hkv, hk = bhk - b * p.Hkv;
  const int k0 = kt * BK;
  const int qt_start = CAUSAL ? max(0, k0 - p.off) / BQ : 0;
  // query tile qt is computed (block mask: the CTA's 128 keys are one mask
  // column, a 64-row query tile half a mask row)
  auto keep = [&](int qt) { return !MASKED || mask_keep(p.bmask, p.nkb, qt >> 1, kt); };
  const int n_iter = p.G * count_kept<MASKED>(keep, qt_start, p.n_qtiles);  // (query head, query tile) iterations
  const WaitGuard g{&abort_flag, p.status, p.limit_ns};

  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(smem_u32(&bar_vready), NCT);
    for (int s = 0; s < ST; ++s) {
      mbar_init(smem_u32(&bar_stfull[s]), 33);  // TMA expect_tx arrive + 32 producer lanes
      mbar_init(smem_u32(&bar_stempty[s]), 1);  // the MMA warp's last read of the stage (dK)
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&bar_dpfull[i]), 1);
      mbar_init(smem_u32(&bar_dsready[i]), NCT);
      mbar_init(smem_u32(&xb.pfull[i]), 1);
      mbar_arrive_expect_tx(smem_u32(&xb.pfull[i]), PtXch::SLOT_BYTES);  // first use of slot i
    }
    mbar_init(smem_u32(&bar_accdone), 1);
    fence_mbar_init();
  }
  if (warp == Gm::MMA_WARP) {
    tmem_alloc(smem_u32(&tmem_slot), Gm::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  cluster_sync_all();  // both CTAs' mbarriers are initialised before any remote arrival
  tc_fence_after_sync();
  const uint32_t tmem = tmem_slot;

  if (warp == Gm::PRODUCER_WARP) {
    // ---------------- producer (whole warp) ----------------
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmdO);
    }
    __syncwarp();
    RingPos<ST> st;
    auto qw = kept_walk<MASKED>(keep, p.n_qtiles);
    int gi = 0, qtile = qw.first(qt_start);  // query head in the group and query tile of iteration it
    // the per-query values of an iteration are loaded one iteration ahead, so
    // their latency overlaps the wait for a free stage
    float pre[BQ / 32];
    auto load_pre = [&]() {
      const int zq = b * p.Hq + hk * p.G + gi;
#pragma unroll
      for (int t = 0; t < BQ / 32; ++t) {
        const int qi = qtile * BQ + lane + 32 * t;
        pre[t] = qi < p.Lq ? p.delta[static_cast<size_t>(zq) * p.Lq + qi] : 0.f;
      }
    };
    if (n_iter > 0) load_pre();
    for (int it = 0; it < n_iter; ++it, st.next()) {
      const int s = st.slot;
      if (it >= ST) mbar_wait(smem_u32(&bar_stempty[s]), st.phase ^ 1u, g, kDevTimeoutBase + 111);
      __syncwarp();
      const int q0 = qtile * BQ;
      const int zq = b * p.Hq + hk * p.G + gi;
      mbar_arrive_expect_tx_w(smem_u32(&bar_stfull[s]), 2 * Gm::Q_BYTES);
      for (int c = 0; c < NCH; ++c) {
        tma_load_3d_w(sQ0 + s * Gm::Q_BYTES + c * BQ * 128, &tmQ, smem_u32(&bar_stfull[s]), c * 64, q0, zq);
        tma_load_3d_w(sdO0 + s * Gm::Q_BYTES + c * BQ * 128, &tmdO, smem_u32(&bar_stfull[s]), c * 64, q0, zq);
      }
#pragma unroll
      for (int t = 0; t < BQ / 32; ++t) dlt_s[s][lane + 32 * t] = pre[t];
      mbar_arrive(smem_u32(&bar_stfull[s]));
      qtile = qw.next(qtile);
      if (qtile >= p.n_qtiles) qtile = qw.first(qt_start), ++gi;
      if (it + 1 < n_iter) load_pre();
    }
    for (int it = (n_iter > ST ? n_iter - ST : 0); it < n_iter; ++it)
      mbar_wait_drain(smem_u32(&bar_stfull[it % ST]), (it / ST) & 1, p.limit_ns);
  } else if (warp == Gm::MMA_WARP) {
    // ---------------- MMA issuer ----------------
    constexpr uint32_t IDESC_DP = make_idesc_f16(128, BQ, BF16, false, false);
    constexpr uint32_t IDESC_ACC = make_idesc_f16(128, D, BF16, false, true);
    const uint64_t dOk = make_sdesc_sw128(sdO0, 16, 1024);       // dO stage 0, K-major
    const uint64_t dQm = make_sdesc_sw128(sQ0, BQ * 128, 1024);  // Q stage 0, MN-major
    RingPos<ST> st, st_d;  // stages of the next dK and of the next dP^T
    // dP^T(it) = V dO^T into buffer it & 1 (V from tensor memory)
    auto issue_dp = [&](int it) {
      const int s = st_d.slot;
      mbar_wait(smem_u32(&bar_stfull[s]), st_d.phase, g, kDevTimeoutBase + 113);
      __syncwarp();
      tc_fence_after_sync();
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t qo = s * Gm::Q_BYTES + (kk >> 2) * (BQ * 128) + (kk & 3) * 32;
        mma_ts_w(tmem + Gm::DPT_COL + (it & 1) * BQ, tmem + Gm::V_COL + kk * 8, sdesc_add(dOk, qo), IDESC_DP,
                 kk > 0 ? 1u : 0u);
      }
      mma_commit_w(smem_u32(&bar_dpfull[it & 1]));
      st_d.next();
    };
    mbar_wait(smem_u32(&bar_vready), 0, g, kDevTimeoutBase + 112);
    for (int it = 0; it < 2 && it < n_iter; ++it) issue_dp(it);
    for (int it = 0; it < n_iter; ++it, st.next()) {
      const int s = st.slot, buf = it & 1;
      // dS^T(it) is in dP^T buffer buf
      mbar_wait(smem_u32(&bar_dsready[buf]), (it >> 1) & 1, g, kDevTimeoutBase + 114);
      __syncwarp();
      tc_fence_after_sync();
      // A operand: queries 32h..32h+31 of warpgroup h as pairs in columns
      // 32h..32h+15 of the buffer
#pragma unroll
      for (int kk = 0; kk < BQ / 16; ++kk) {
        const uint32_t acol = Gm::DPT_COL + buf * BQ + (kk >> 1) * 32 + (kk & 1) * 8;
        mma_ts_w(tmem + Gm::DK_COL, tmem + acol, sdesc_add(dQm, s * Gm::Q_BYTES + kk * 2048), IDESC_ACC,
                 (it > 0 || kk > 0) ? 1u : 0u);
      }
      // dP^T(it) and dK(it) were this thread's reads of the stage
      mma_commit_w(smem_u32(&bar_stempty[s]));
      // dP^T(it+2) overwrites dS^T(it) behind the dK MMAs that read it
      if (it + 2 < n_iter) issue_dp(it + 2);
    }
    mma_commit_w(smem_u32(&bar_accdone));
    mbar_wait_drain(smem_u32(&bar_accdone), 0, p.limit_ns);
    __syncwarp();
  } else {
    // ---------------- key-row threads ----------------
    const int quad = warp & 3;   // TMEM lane quadrant (key rows)
    const int half = warp >> 2;  // query columns 32*half .. +31; V / dK columns half*128 .. +127
    const int r = quad * 32 + lane;
    const int kj = k0 + r;
    const uint32_t lrow = static_cast<uint32_t>(quad * 32) << 16;
    {
      // V row into tensor memory: this thread copies elements [half*128, half*128+128)
      // of value row kj (zeros past Lk) as 64 columns of 16-bit pairs.
      const uint4* src = reinterpret_cast<const uint4*>(reinterpret_cast<const typename E::T*>(p.v) +
                                                        (static_cast<size_t>(bhk) * p.kv_pitch + kj) * D + half * 128);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t t16[16];
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          uint4 x = make_uint4(0u, 0u, 0u, 0u);
          if (kj < p.Lk) x = src[c * 4 + v];
          t16[4 * v + 0] = x.x, t16[4 * v + 1] = x.y, t16[4 * v + 2] = x.z, t16[4 * v + 3] = x.w;
        }
        tmem_st16(tmem + lrow + Gm::V_COL + half * 64 + c * 16, t16);
      }
      tmem_st_wait();
      tc_fence_before_sync();
      mbar_arrive(smem_u32(&bar_vready));
    }
    RingPos<ST> st;
    for (int it = 0; it < n_iter; ++it, st.next()) {
      const int s = st.slot, buf = it & 1;
      mbar_wait(smem_u32(&bar_stfull[s]), st.phase, g, kDevTimeoutBase + 115);
      mbar_wait(smem_u32(&bar_dpfull[buf]), (it >> 1) & 1, g, kDevTimeoutBase + 116);
      __syncwarp();
      tc_fence_after_sync();
      const uint32_t dcol = tmem + lrow + Gm::DPT_COL + buf * BQ + half * 32;
      uint32_t dr[32];
      tmem_ld32(dcol, dr);
      // P^T(it) from the dV CTA: 32 queries (four chunks) of this thread's key row
      mbar_wait(smem_u32(&xb.pfull[buf]), (it >> 1) & 1, g, kDevTimeoutBase + 117);
      // the slot's next use (query tile it + 2) expects its bytes: the dV CTA
      // cannot write them before every warp here has released this use
      if (threadIdx.x == 0 && it + 2 < n_iter && !abort_flag) mbar_arrive_expect_tx(smem_u32(&xb.pfull[buf]), PtXch::SLOT_BYTES);
      uint4 pv[4];
#pragma unroll
      for (int v = 0; v < 4; ++v) pv[v] = ld_shared_v4(PtXch::addr(sX, buf, r, half * 4 + v));
      tmem_ld_wait(dr);
      const uint64_t* dlt_row = reinterpret_cast<const uint64_t*>(&dlt_s[s][half * 32]);
      const uint32_t pw[16] = {pv[0].x, pv[0].y, pv[0].z, pv[0].w, pv[1].x, pv[1].y, pv[1].z, pv[1].w,
                               pv[2].x, pv[2].y, pv[2].z, pv[2].w, pv[3].x, pv[3].y, pv[3].z, pv[3].w};
      uint32_t dk[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int c0 = 2 * i;
        const float2 pp = E::unpack(pw[i]);
        const uint64_t d2 = f2_sub(f2_pack(__uint_as_float(dr[c0]), __uint_as_float(dr[c0 + 1])), dlt_row[i]);
        float ds0, ds1;
        f2_unpack(f2_mul(f2_pack(pp.x, pp.y), d2), ds0, ds1);
        dk[i] = E::pack(ds0, ds1);
      }
      // the warp has used its values of the slot: it may be refilled
      __syncwarp();
      if (lane == 0) mbar_arrive_remote(cluster_map(smem_u32(&xb.pfree[buf]), 0));
      tmem_st16(dcol, dk);
      tmem_st_wait();
      tc_fence_before_sync();
      mbar_arrive(smem_u32(&bar_dsready[buf]));
    }
    mbar_wait(smem_u32(&bar_accdone), 0, g, kDevTimeoutBase + 118);
    __syncwarp();
    tc_fence_after_sync();
    // epilogue: warpgroup `half` writes dK columns [half*128, half*128+128)
    typename E::T* dst = reinterpret_cast<typename E::T*>(p.dk) + (static_cast<size_t>(bhk) * p.Lk + kj) * D;
#pragma unroll 1
    for (int c = half * 4; c < half * 4 + 4; ++c) {
      uint32_t rr[32];
      if (n_iter > 0) {  // the same for the whole CTA: tcgen05.ld is warp-collective
        tmem_ld32(tmem + lrow + Gm::DK_COL + c * 32, rr);
        tmem_ld_wait(rr);
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) rr[i] = 0u;  // no kept query tile: dK = 0
      }
      if (kj < p.Lk) store_row32<BF16>(dst + c * 32, rr, p.scale);
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == Gm::MMA_WARP) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, Gm::TMEM_COLS);
  }
}

// D = 256, dV half (cluster rank 0): K in tensor memory as the A operand of
// S^T = K Q^T (copied in by the row threads), so shared memory holds only
// Q/dO stages (three of 64 KB, enough to hide the loads' latency).  Tensor
// memory: dV (256 columns), K (128), S^T (two buffers of 64).  The row threads
// turn S^T into P^T (16-bit pairs), write it over the columns they read and
// into the partner CTA's hand-off slot, and the MMA warp issues dV += P^T dO,
// then S^T of the tile after next into the same buffer.
struct Dv256Geom {
  static constexpr int D = 256, BK = 128, BQ = 64, NCH = 4;
  static constexpr int Q_BYTES = NCH * BQ * 128;  // 32 KB
  static constexpr int STAGES_FIT = (kMaxDynSmem - kSmemReserve - 1024) / (2 * Q_BYTES);
  static constexpr int STAGES = STAGES_FIT > 3 ? 3 : STAGES_FIT;
  static constexpr int SMEM_BYTES = 1024 + STAGES * 2 * Q_BYTES;
  static constexpr int DV_COL = 0, K_COL = 256, ST_COL = 384;  // S^T: 2 x 64
  static constexpr int TMEM_COLS = 512;
  static constexpr int NUM_COMPUTE_WARPS = 8;
  static constexpr int NCT = 32 * NUM_COMPUTE_WARPS;
  static constexpr int PRODUCER_WARP = NUM_COMPUTE_WARPS;
  static constexpr int MMA_WARP = NUM_COMPUTE_WARPS + 1;
  static constexpr int NUM_THREADS = 32 * (NUM_COMPUTE_WARPS + 2);
  static_assert(STAGES >= 3, "three Q/dO stages");
  static_assert(ST_COL + 2 * BQ <= TMEM_COLS, "tensor memory budget");
};

template <bool BF16, bool CAUSAL, bool MASKED>
__device__ __forceinline__ void dv256_tile(const CUtensorMap& tmQ, const CUtensorMap& tmdO, const BwdParams& p,
                                           const int bhk, const int kt, PtXchBars& xb) {
  using Gm = Dv256Geom;
  using E = Elem<BF16>;
  constexpr int D = Gm::D, BQ = Gm::BQ, BK = Gm::BK, NCH = Gm::NCH, ST = Gm::STAGES, NCT = Gm::NCT;

  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t bar_kready, bar_stfull[ST], bar_stempty[ST], bar_sfull[2], bar_pready[2], bar_accdone;
  __shared__ __align__(16) float nlse_s[ST][BQ];  // -lse per query column
  __shared__ uint32_t tmem_slot;
  __shared__ volatile int abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t sQ0 = sbase;
  const uint32_t sdO0 = sQ0 + ST * Gm::Q_BYTES;

  const int b = bhk / p.Hkv, hk = bhk - b * p.Hkv;
  const int k0 = kt * BK;
  const int qt_start = CAUSAL ? max(0, k0 - p.off) / BQ : 0;
  // query tile qt is computed (block mask: the CTA's 128 keys are one mask
  // column, a 64-row query tile half a mask row)
  auto keep = [&](int qt) { return !MASKED || mask_keep(p.bmask, p.nkb, qt >> 1, kt); };
  const int n_iter = p.G * count_kept<MASKED>(keep, qt_start, p.n_qtiles);  // (query head, query tile) iterations
  const WaitGuard g{&abort_flag, p.status, p.limit_ns};

  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(smem_u32(&bar_kready), NCT);
    for (int s = 0; s < ST; ++s) {
      mbar_init(smem_u32(&bar_stfull[s]), 33);  // TMA expect_tx arrive + 32 producer lanes
      mbar_init(smem_u32(&bar_stempty[s]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&bar_sfull[i]), 1);
      mbar_init(smem_u32(&bar_pready[i]), NCT);
      mbar_init(smem_u32(&xb.pfree[i]), Dk256Geom::NUM_COMPUTE_WARPS);  // the dK CTA's row warps
    }
    mbar_init(smem_u32(&bar_accdone), 1);
    fence_mbar_init();
  }
  if (warp == Gm::MMA_WARP) {
    tmem_alloc(smem_u32(&tmem_slot), Gm::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  cluster_sync_all();  // both CTAs' mbarriers are initialised before any remote arrival
  tc_fence_after_sync();
  const uint32_t tmem = tmem_slot;

  if (warp == Gm::PRODUCER_WARP) {
    // ---------------- producer (whole warp) ----------------
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmdO);
    }
    __syncwarp();
    RingPos<ST> st;
    auto qw = kept_walk<MASKED>(keep, p.n_qtiles);
    int gi = 0, qtile = qw.first(qt_start);
    // the per-query values of an iteration are loaded one iteration ahead, so
    // their latency overlaps the wait for a free stage
    float pre[BQ / 32];
    auto load_pre = [&]() {
      const int zq = b * p.Hq + hk * p.G + gi;
#pragma unroll
      for (int t = 0; t < BQ / 32; ++t) {
        const int qi = qtile * BQ + lane + 32 * t;
        pre[t] = qi < p.Lq ? -p.lse[static_cast<size_t>(zq) * p.Lq + qi] : -INFINITY;
      }
    };
    if (n_iter > 0) load_pre();
    for (int it = 0; it < n_iter; ++it, st.next()) {
      const int s = st.slot;
      if (it >= ST) mbar_wait(smem_u32(&bar_stempty[s]), st.phase ^ 1u, g, kDevTimeoutBase + 131);
      __syncwarp();
      const int q0 = qtile * BQ;
      const int zq = b * p.Hq + hk * p.G + gi;
      mbar_arrive_expect_tx_w(smem_u32(&bar_stfull[s]), 2 * Gm::Q_BYTES);
      for (int c = 0; c < NCH; ++c) {
        tma_load_3d_w(sQ0 + s * Gm::Q_BYTES + c * BQ * 128, &tmQ, smem_u32(&bar_stfull[s]), c * 64, q0, zq);
        tma_load_3d_w(sdO0 + s * Gm::Q_BYTES + c * BQ * 128, &tmdO, smem_u32(&bar_stfull[s]), c * 64, q0, zq);
      }
#pragma unroll
      for (int t = 0; t < BQ / 32; ++t) nlse_s[s][lane + 32 * t] = pre[t];
      mbar_arrive(smem_u32(&bar_stfull[s]));
      qtile = qw.next(qtile);
      if (qtile >= p.n_qtiles) qtile = qw.first(qt_start), ++gi;
      if (it + 1 < n_iter) load_pre();
    }
    for (int it = (n_iter > ST ? n_iter - ST : 0); it < n_iter; ++it)
      mbar_wait_drain(smem_u32(&bar_stfull[it % ST]), (it / ST) & 1, p.limit_ns);
  } else if (warp == Gm::MMA_WARP) {
    // ---------------- MMA issuer ----------------
    constexpr uint32_t IDESC_S = make_idesc_f16(128, BQ, BF16, false, false);
    constexpr uint32_t IDESC_ACC = make_idesc_f16(128, D, BF16, false, true);
    const uint64_t dQk = make_sdesc_sw128(sQ0, 16, 1024);         // Q stage 0, K-major
    const uint64_t dOm = make_sdesc_sw128(sdO0, BQ * 128, 1024);  // dO stage 0, MN-major
    RingPos<ST> st, st_s;  // stages of the next dV and of the next S^T
    auto issue_s = [&](int it) {
      const int s = st_s.slot;
      mbar_wait(smem_u32(&bar_stfull[s]), st_s.phase, g, kDevTimeoutBase + 132);
      __syncwarp();
      tc_fence_after_sync();
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t qo = s * Gm::Q_BYTES + (kk >> 2) * (BQ * 128) + (kk & 3) * 32;
        mma_ts_w(tmem + Gm::ST_COL + (it & 1) * BQ, tmem + Gm::K_COL + kk * 8, sdesc_add(dQk, qo), IDESC_S,
                 kk > 0 ? 1u : 0u);
      }
      mma_commit_w(smem_u32(&bar_sfull[it & 1]));
      st_s.next();
    };
    mbar_wait(smem_u32(&bar_kready), 0, g, kDevTimeoutBase + 133);
    for (int it = 0; it < 2 && it < n_iter; ++it) issue_s(it);
    for (int it = 0; it < n_iter; ++it, st.next()) {
      const int s = st.slot, buf = it & 1;
      mbar_wait(smem_u32(&bar_pready[buf]), (it >> 1) & 1, g, kDevTimeoutBase + 134);
      __syncwarp();
      tc_fence_after_sync();
      // A operand: queries 32h..32h+31 of warpgroup h as pairs in columns
      // 32h..32h+15 of the buffer
#pragma unroll
      for (int kk = 0; kk < BQ / 16; ++kk) {
        const uint32_t acol = Gm::ST_COL + buf * BQ + (kk >> 1) * 32 + (kk & 1) * 8;
        mma_ts_w(tmem + Gm::DV_COL, tmem + acol, sdesc_add(dOm, s * Gm::Q_BYTES + kk * 2048), IDESC_ACC,
                 (it > 0 || kk > 0) ? 1u : 0u);
      }
      mma_commit_w(smem_u32(&bar_stempty[s]));
      // S^T(it+2) overwrites P^T(it) behind the dV MMAs that read it
      if (it + 2 < n_iter) issue_s(it + 2);
    }
    mma_commit_w(smem_u32(&bar_accdone));
    mbar_wait_drain(smem_u32(&bar_accdone), 0, p.limit_ns);
    __syncwarp();
  } else {
    // ---------------- key-row threads ----------------
    const int quad = warp & 3;
    const int half = warp >> 2;  // query columns 32*half .. +31; K / dV columns half*128 .. +127
    const int r = quad * 32 + lane;
    const int kj = k0 + r;
    const uint32_t lrow = static_cast<uint32_t>(quad * 32) << 16;
    const uint64_t sl2x2 = f2_pack(p.scale_log2, p.scale_log2);
    const int qmin = kj - p.off;
    const uint32_t sX1 = cluster_map(sbase + Dk256Geom::XCH_OFF, 1);  // the dK CTA's hand-off slots
    {
      const uint4* src = reinterpret_cast<const uint4*>(reinterpret_cast<const typename E::T*>(p.k) +
                                                        (static_cast<size_t>(bhk) * p.kv_pitch + kj) * D + half * 128);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t t16[16];
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          uint4 x = make_uint4(0u, 0u, 0u, 0u);
          if (kj < p.Lk) x = src[c * 4 + v];
          t16[4 * v + 0] = x.x, t16[4 * v + 1] = x.y, t16[4 * v + 2] = x.z, t16[4 * v + 3] = x.w;
        }
        tmem_st16(tmem + lrow + Gm::K_COL + half * 64 + c * 16, t16);
      }
      tmem_st_wait();
      tc_fence_before_sync();
      mbar_arrive(smem_u32(&bar_kready));
    }
    RingPos<ST> st;
    auto qw = kept_walk<MASKED>(keep, p.n_qtiles);
    int qtile = qw.first(qt_start);
    for (int it = 0; it < n_iter; ++it, st.next()) {
      const int s = st.slot, buf = it & 1;
      const int q0 = qtile * BQ;
      qtile = qw.next(qtile);
      if (qtile >= p.n_qtiles) qtile = qw.first(qt_start);
      mbar_wait(smem_u32(&bar_stfull[s]), st.phase, g, kDevTimeoutBase + 135);
      mbar_wait(smem_u32(&bar_sfull[buf]), (it >> 1) & 1, g, kDevTimeoutBase + 136);
      __syncwarp();
      tc_fence_after_sync();
      const uint32_t scol = tmem + lrow + Gm::ST_COL + buf * BQ + half * 32;
      uint32_t sr[32];
      tmem_ld32(scol, sr);
      tmem_ld_wait(sr);
      const bool need_mask = CAUSAL && (q0 < k0 + BK - 1 - p.off);
      const uint64_t* nlse_row = reinterpret_cast<const uint64_t*>(&nlse_s[s][half * 32]);
      const int qc0 = q0 + half * 32;
      uint32_t pk[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int c0 = 2 * i;
        float x0, x1;
        f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[c0]), __uint_as_float(sr[c0 + 1])), sl2x2, nlse_row[i]), x0, x1);
        float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
        if (need_mask) {
          if (qc0 + c0 < qmin) p0 = 0.f;
          if (qc0 + c0 + 1 < qmin) p1 = 0.f;
        }
        pk[i] = E::pack(p0, p1);
      }
      tmem_st16(scol, pk);
      // P^T(it) to the dK CTA: four 16-byte chunks of this thread's key row,
      // once that CTA has used the slot's previous contents
      if (it >= 2) mbar_wait(smem_u32(&xb.pfree[buf]), ((it >> 1) & 1) ^ 1, g, kDevTimeoutBase + 138);
      const uint32_t full1 = cluster_map(smem_u32(&xb.pfull[buf]), 1);
#pragma unroll
      for (int v = 0; v < 4; ++v)
        st_async_v4(PtXch::addr(sX1, buf, r, half * 4 + v), pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3],
                    full1);
      tmem_st_wait();
      tc_fence_before_sync();
      mbar_arrive(smem_u32(&bar_pready[buf]));
    }
    mbar_wait(smem_u32(&bar_accdone), 0, g, kDevTimeoutBase + 137);
    __syncwarp();
    tc_fence_after_sync();
    typename E::T* dst = reinterpret_cast<typename E::T*>(p.dv) + (static_cast<size_t>(bhk) * p.Lk + kj) * D;
#pragma unroll 1
    for (int c = half * 4; c < half * 4 + 4; ++c) {
      uint32_t rr[32];
      if (n_iter > 0) {
        tmem_ld32(tmem + lrow + Gm::DV_COL + c * 32, rr);
        tmem_ld_wait(rr);
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) rr[i] = 0u;  // no kept query tile: dV = 0
      }
      if (kj < p.Lk) store_row32<BF16>(dst + c * 32, rr, 1.f);
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == Gm::MMA_WARP) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, Gm::TMEM_COLS);
  }
}

// D = 256: both halves in one launch, as the two CTAs of a cluster:
// x = 2 * (b * Hkv + hk) + (0: dV, 1: dK), y = key tile.  Clusters are
// dispatched in x-then-y order, so the heavy key tiles (small kt: the most
// visible query tiles under causal masking) start first.
struct DkvPairGeom {
  static_assert(Dv256Geom::NUM_THREADS == Dk256Geom::NUM_THREADS, "one block size for both halves");
  static constexpr int NUM_THREADS = Dk256Geom::NUM_THREADS;
  static constexpr int SMEM_BYTES =
      Dv256Geom::SMEM_BYTES > Dk256Geom::SMEM_BYTES ? Dv256Geom::SMEM_BYTES : Dk256Geom::SMEM_BYTES;
  static constexpr int BQ = Dk256Geom::BQ, BK = Dk256Geom::BK;
  static_assert(Dv256Geom::BQ == BQ && Dv256Geom::BK == BK, "one tiling for both halves");
};

// MASKED: block-sparse variant; both CTAs of a key tile walk the query tiles
// its mask column keeps and write zeros if it keeps none.
template <bool BF16, bool CAUSAL, bool MASKED = false>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(DkvPairGeom::NUM_THREADS, 1)
    attn_bwd_dkv_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmdO,
                        const BwdParams p) {
  __shared__ PtXchBars xb;
  const int bhk = static_cast<int>(blockIdx.x >> 1), kt = static_cast<int>(blockIdx.y);
  if (cluster_ctarank() == 1)
    dk256_tile<BF16, CAUSAL, MASKED>(tmQ, tmdO, p, bhk, kt, xb);
  else
    dv256_tile<BF16, CAUSAL, MASKED>(tmQ, tmdO, p, bhk, kt, xb);
  // neither CTA leaves while the other may still write its shared memory
  cluster_sync_all();
}

}  // namespace gbattn
