// Backward, dK/dV kernel: owns a tile of BK = 128 key rows of one (batch, KV
// head) and loops over the G query heads of its group, then over the visible
// query tiles ("feat(attention): complete Flash Attention VJP implementation",
// section "Two-Kernel Design": grid [NK, kvH, B], loop over the GQA group then
// the Q blocks, K-row ownership so dK and dV need no atomics).  Per query tile
// everything is computed transposed, so the key row is the TMEM lane:
//   S^T = K Q^T, dP^T = V dO^T                       (tcgen05, fp32 in TMEM)
//   P^T = exp2(S^T * scale_log2 - lse), dS^T = P^T * (dP^T - delta)
//   dV += P^T dO, dK += dS^T Q                        (tcgen05, A from TMEM)
// and finally dK is scaled by `scale`.
//
// MODE selects which outputs one CTA accumulates.  kDkvBoth keeps dK and dV
// in tensor memory together (D <= 128).  At D = 256 the two accumulators
// alone fill the 512 TMEM columns, so dV (kDkvDvOnly: S^T, P^T, dV) and dK
// (kDkvDkOnly: S^T, dP^T, dS^T, dK) are produced by separate CTAs.
//
// Warp roles (192 threads): warps 0-3 key-row threads, warp 4 producer (TMA
// for Q/dO tiles, plain loads for the per-query lse/delta values), warp 5 MMA
// issuer and TMEM owner.
#pragma once

#include "kernel_common.cuh"

namespace gbattn {

enum DkvMode : int { kDkvBoth = 0, kDkvDvOnly = 1, kDkvDkOnly = 2 };

template <int D, int MODE>
struct DkvGeom {
  static constexpr int BK = 128;  // key rows per CTA (MMA M)
  static constexpr int BQ = 64;   // query rows per iteration (MMA N of S^T)
  static constexpr int NCH = n_chunks(D);
  static constexpr bool NEED_V = MODE != kDkvDvOnly;   // dP^T needs V
  static constexpr bool NEED_DS = MODE != kDkvDvOnly;  // dK path
  static constexpr bool NEED_DV = MODE != kDkvDkOnly;  // dV path
  static constexpr int K_BYTES = NCH * BK * 128;
  static constexpr int Q_BYTES = NCH * BQ * 128;
  static constexpr int RES_BYTES = K_BYTES * (NEED_V ? 2 : 1);
  static constexpr int STAGES_FIT = (kMaxDynSmem - kSmemReserve - 1024 - RES_BYTES) / (2 * Q_BYTES);
  static constexpr int STAGES = STAGES_FIT > 4 ? 4 : STAGES_FIT;
  static constexpr int SMEM_BYTES = 1024 + RES_BYTES + STAGES * 2 * Q_BYTES;
  static constexpr int ACC_W = (D <= 128) ? 128 : 256;
  static constexpr int DK_COL = 0;
  static constexpr int DV_COL = (MODE == kDkvBoth) ? ACC_W : 0;
  static constexpr int ST_COL = (MODE == kDkvBoth) ? 2 * ACC_W : ACC_W;
  static constexpr int DPT_COL = ST_COL + BQ;                      // unused in DvOnly
  static constexpr int PT_COL = (MODE == kDkvDvOnly) ? ST_COL + BQ : DPT_COL + BQ;
  static constexpr int DST_COL = (MODE == kDkvDkOnly) ? DPT_COL + BQ : PT_COL + BQ / 2;
  static constexpr int TMEM_COLS = 512;
  static constexpr int NUM_THREADS = 192;
  static_assert(STAGES >= 1, "shared memory budget");
  static_assert(MODE != kDkvBoth || D <= 128, "dK and dV together need D <= 128");
  static_assert(DST_COL + BQ / 2 <= TMEM_COLS && PT_COL + BQ / 2 <= TMEM_COLS, "tensor memory budget");
};

template <int D, bool BF16, bool CAUSAL, int MODE>
__global__ void __launch_bounds__(192, 1)
    attn_bwd_dkv_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                        const BwdParams p) {
  using Gm = DkvGeom<D, MODE>;
  using E = Elem<BF16>;
  constexpr int BQ = Gm::BQ, BK = Gm::BK, NCH = Gm::NCH, ST = Gm::STAGES;

  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t bar_kv, bar_stfull[ST], bar_stempty[ST], bar_sfull, bar_pready, bar_accdone;
  __shared__ float lse_s[ST][BQ], dlt_s[ST][BQ];
  __shared__ uint32_t tmem_slot;
  __shared__ volatile int abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t sK = sbase;
  const uint32_t sV = sK + Gm::K_BYTES;  // only when NEED_V
  const uint32_t sQ0 = sbase + Gm::RES_BYTES;
  const uint32_t sdO0 = sQ0 + ST * Gm::Q_BYTES;

  const int bhk = blockIdx.x;  // b * Hkv + hk
  const int b = bhk / p.Hkv, hk = bhk - b * p.Hkv;
  const int kt = blockIdx.y;
  const int k0 = kt * BK;
  const int qt_start = CAUSAL ? max(0, k0 - p.off) / BQ : 0;
  const int nq = p.n_qtiles - qt_start;
  const int n_iter = p.G * nq;
  const WaitGuard g{&abort_flag, p.status, p.limit_ns};

  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(smem_u32(&bar_kv), 1);
    for (int s = 0; s < ST; ++s) {
      mbar_init(smem_u32(&bar_stfull[s]), 33);  // TMA expect_tx arrive + 32 producer lanes
      mbar_init(smem_u32(&bar_stempty[s]), 1);
    }
    mbar_init(smem_u32(&bar_sfull), 1);
    mbar_init(smem_u32(&bar_pready), 128);
    mbar_init(smem_u32(&bar_accdone), 1);
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc(smem_u32(&tmem_slot), Gm::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = tmem_slot;

  if (warp == 4) {
    // ---------------- producer (whole warp) ----------------
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmdO);
      if (Gm::NEED_V) tma_prefetch_desc(&tmV);
      mbar_arrive_expect_tx(smem_u32(&bar_kv), Gm::RES_BYTES);
      for (int c = 0; c < NCH; ++c) {
        tma_load_3d(sK + c * BK * 128, &tmK, smem_u32(&bar_kv), c * 64, k0, bhk);
        if (Gm::NEED_V) tma_load_3d(sV + c * BK * 128, &tmV, smem_u32(&bar_kv), c * 64, k0, bhk);
      }
    }
    for (int it = 0; it < n_iter; ++it) {
      const int s = it % ST, u = it / ST;
      if (u > 0) mbar_wait(smem_u32(&bar_stempty[s]), (u - 1) & 1, g, kDevTimeoutBase + 21);
      const int gi = it / nq;
      const int q0 = (qt_start + (it - gi * nq)) * BQ;
      const int zq = b * p.Hq + hk * p.G + gi;
      if (lane == 0) {
        mbar_arrive_expect_tx(smem_u32(&bar_stfull[s]), 2 * Gm::Q_BYTES);
        for (int c = 0; c < NCH; ++c) {
          tma_load_3d(sQ0 + s * Gm::Q_BYTES + c * BQ * 128, &tmQ, smem_u32(&bar_stfull[s]), c * 64, q0, zq);
          tma_load_3d(sdO0 + s * Gm::Q_BYTES + c * BQ * 128, &tmdO, smem_u32(&bar_stfull[s]), c * 64, q0,
                      zq);
        }
      }
#pragma unroll
      for (int t = 0; t < BQ / 32; ++t) {
        const int c = lane + 32 * t;
        const int qi = q0 + c;
        const size_t row = static_cast<size_t>(zq) * p.Lq + qi;
        lse_s[s][c] = qi < p.Lq ? p.lse[row] : INFINITY;
        dlt_s[s][c] = (Gm::NEED_DS && qi < p.Lq) ? p.delta[row] : 0.f;
      }
      mbar_arrive(smem_u32(&bar_stfull[s]));
    }
    for (int it = (n_iter > ST ? n_iter - ST : 0); it < n_iter; ++it)
      mbar_wait_drain(smem_u32(&bar_stfull[it % ST]), (it / ST) & 1, p.limit_ns);
  } else if (warp == 5) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      constexpr uint32_t IDESC_S = make_idesc_f16(128, BQ, BF16, false, false);
      constexpr uint32_t IDESC_ACC = make_idesc_f16(128, D, BF16, false, true);
      mbar_wait(smem_u32(&bar_kv), 0, g, kDevTimeoutBase + 22);
      tc_fence_after_sync();
      for (int it = 0; it < n_iter; ++it) {
        const int s = it % ST;
        const uint32_t qb = sQ0 + s * Gm::Q_BYTES, ob = sdO0 + s * Gm::Q_BYTES;
        mbar_wait(smem_u32(&bar_stfull[s]), (it / ST) & 1, g, kDevTimeoutBase + 23);
        tc_fence_after_sync();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t ko = (kk >> 2) * (BK * 128) + (kk & 3) * 32;
          const uint32_t qo = (kk >> 2) * (BQ * 128) + (kk & 3) * 32;
          mma_ss(tmem + Gm::ST_COL, make_sdesc_sw128(sK + ko, 16, 1024), make_sdesc_sw128(qb + qo, 16, 1024),
                 IDESC_S, kk > 0 ? 1u : 0u);
        }
        if (Gm::NEED_DS) {
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t ko = (kk >> 2) * (BK * 128) + (kk & 3) * 32;
            const uint32_t qo = (kk >> 2) * (BQ * 128) + (kk & 3) * 32;
            mma_ss(tmem + Gm::DPT_COL, make_sdesc_sw128(sV + ko, 16, 1024),
                   make_sdesc_sw128(ob + qo, 16, 1024), IDESC_S, kk > 0 ? 1u : 0u);
          }
        }
        mma_commit(smem_u32(&bar_sfull));
        mbar_wait(smem_u32(&bar_pready), it & 1, g, kDevTimeoutBase + 24);
        tc_fence_after_sync();
        if (Gm::NEED_DV) {
#pragma unroll
          for (int kk = 0; kk < BQ / 16; ++kk)
            mma_ts(tmem + Gm::DV_COL, tmem + Gm::PT_COL + kk * 8,
                   make_sdesc_sw128(ob + kk * 2048, BQ * 128, 1024), IDESC_ACC, (it > 0 || kk > 0) ? 1u : 0u);
        }
        if (Gm::NEED_DS) {
#pragma unroll
          for (int kk = 0; kk < BQ / 16; ++kk)
            mma_ts(tmem + Gm::DK_COL, tmem + Gm::DST_COL + kk * 8,
                   make_sdesc_sw128(qb + kk * 2048, BQ * 128, 1024), IDESC_ACC, (it > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(smem_u32(&bar_stempty[s]));
      }
      mma_commit(smem_u32(&bar_accdone));
      mbar_wait_drain(smem_u32(&bar_accdone), 0, p.limit_ns);
    }
  } else {
    // ---------------- key-row threads ----------------
    const int r = warp * 32 + lane;
    const int kj = k0 + r;
    const uint32_t lrow = static_cast<uint32_t>(warp * 32) << 16;
    const float sl2 = p.scale_log2;
    const int qmin = kj - p.off;  // causal: queries below this index cannot see key kj
    for (int it = 0; it < n_iter; ++it) {
      const int s = it % ST;
      const int gi = it / nq;
      const int q0 = (qt_start + (it - gi * nq)) * BQ;
      mbar_wait(smem_u32(&bar_stfull[s]), (it / ST) & 1, g, kDevTimeoutBase + 25);
      mbar_wait(smem_u32(&bar_sfull), it & 1, g, kDevTimeoutBase + 26);
      __syncwarp();
      tc_fence_after_sync();
      const bool need_mask = CAUSAL && (q0 < k0 + BK - 1 - p.off);
#pragma unroll
      for (int c = 0; c < BQ / 32; ++c) {
        uint32_t sr[32], dr[32];
        tmem_ld32(tmem + lrow + Gm::ST_COL + c * 32, sr);
        if (Gm::NEED_DS) tmem_ld32(tmem + lrow + Gm::DPT_COL + c * 32, dr);
        tmem_ld_wait(sr);
        if (Gm::NEED_DS) reg_fence(dr);
        uint32_t pk[16], dk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int c0 = c * 32 + 2 * i;
          float p0 = ex2_approx(fmaf(__uint_as_float(sr[2 * i]), sl2, -lse_s[s][c0]));
          float p1 = ex2_approx(fmaf(__uint_as_float(sr[2 * i + 1]), sl2, -lse_s[s][c0 + 1]));
          if (need_mask) {
            if (q0 + c0 < qmin) p0 = 0.f;
            if (q0 + c0 + 1 < qmin) p1 = 0.f;
          }
          pk[i] = E::pack(p0, p1);
          if (Gm::NEED_DS) {
            const float ds0 = p0 * (__uint_as_float(dr[2 * i]) - dlt_s[s][c0]);
            const float ds1 = p1 * (__uint_as_float(dr[2 * i + 1]) - dlt_s[s][c0 + 1]);
            dk[i] = E::pack(ds0, ds1);
          }
        }
        if (Gm::NEED_DV) tmem_st16(tmem + lrow + Gm::PT_COL + c * 16, pk);
        if (Gm::NEED_DS) tmem_st16(tmem + lrow + Gm::DST_COL + c * 16, dk);
      }
      tmem_st_wait();
      tc_fence_before_sync();
      mbar_arrive(smem_u32(&bar_pready));
    }
    mbar_wait(smem_u32(&bar_accdone), 0, g, kDevTimeoutBase + 27);
    __syncwarp();
    tc_fence_after_sync();
    const size_t row = static_cast<size_t>(bhk) * p.Lk + kj;
    if (Gm::NEED_DS) {
      typename E::T* dst = reinterpret_cast<typename E::T*>(p.dk) + row * D;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t rr[32];
        tmem_ld32(tmem + lrow + Gm::DK_COL + c * 32, rr);
        tmem_ld_wait(rr);
        if (kj < p.Lk) store_row32<BF16>(dst + c * 32, rr, p.scale);
      }
    }
    if (Gm::NEED_DV) {
      typename E::T* dst = reinterpret_cast<typename E::T*>(p.dv) + row * D;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t rr[32];
        tmem_ld32(tmem + lrow + Gm::DV_COL + c * 32, rr);
        tmem_ld_wait(rr);
        if (kj < p.Lk) store_row32<BF16>(dst + c * 32, rr, 1.f);
      }
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, Gm::TMEM_COLS);
  }
}

}  // namespace gbattn
