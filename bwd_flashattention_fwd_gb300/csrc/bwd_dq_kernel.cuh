// Backward, dQ kernel: owns a tile of BQ = 128 query rows of one (batch,
// query head) and loops over the visible key tiles ("feat(attention):
// complete Flash Attention VJP implementation", section "Two-Kernel Design":
// the dQ kernel's grid is [NQ, H, B] and its loop runs over KV blocks).  Per
// key tile, with S and dP recomputed on the tensor cores:
//   S = Q K^T, dP = dO V^T                      (tcgen05, fp32 in TMEM)
//   P = exp2(S * scale_log2 - lse), dS = P * (dP - delta)   (row threads)
//   dQ += dS K                                  (tcgen05, dS read from TMEM)
// and finally dQ is scaled by `scale` (section "Background": dS carries the
// softmax scale, dQ = dS K).  No other CTA writes these dQ rows, so no atomics.
//
// Warp roles (192 threads): warps 0-3 row threads (TMEM lane = row), warp 4
// TMA producer, warp 5 MMA issuer and TMEM owner.
#pragma once

#include "kernel_common.cuh"

namespace gbattn {

template <int D>
struct DqGeom {
  static constexpr int BQ = 128;
  static constexpr int BK = (D == 256) ? 64 : 128;
  static constexpr int NCH = n_chunks(D);
  static constexpr int Q_BYTES = NCH * BQ * 128;
  static constexpr int KV_BYTES = NCH * BK * 128;
  static constexpr int STAGES_FIT =
      (kMaxDynSmem - kSmemReserve - 1024 - 2 * Q_BYTES) / (2 * KV_BYTES);
  static constexpr int STAGES = STAGES_FIT > 4 ? 4 : STAGES_FIT;
  static constexpr int SMEM_BYTES = 1024 + 2 * Q_BYTES + STAGES * 2 * KV_BYTES;
  static constexpr int DQ_COL = 0;
  static constexpr int S_COL = (D <= 128) ? 128 : 256;
  static constexpr int DP_COL = S_COL + BK;
  static constexpr int DS_COL = DP_COL + BK;
  static constexpr int TMEM_COLS = 512;
  static constexpr int NUM_THREADS = 192;
  static_assert(STAGES >= 1, "shared memory budget");
  static_assert(DS_COL + BK / 2 <= TMEM_COLS, "tensor memory budget");
};

template <int D, bool BF16, bool CAUSAL>
__global__ void __launch_bounds__(192, 1)
    attn_bwd_dq_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                       const BwdParams p) {
  using Gm = DqGeom<D>;
  using E = Elem<BF16>;
  constexpr int BQ = Gm::BQ, BK = Gm::BK, NCH = Gm::NCH, ST = Gm::STAGES;

  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t bar_q, bar_kfull[ST], bar_vfull[ST], bar_kvempty[ST], bar_sfull, bar_dsready,
      bar_dqdone;
  __shared__ uint32_t tmem_slot;
  __shared__ volatile int abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t sQ = sbase;
  const uint32_t sdO = sQ + Gm::Q_BYTES;
  const uint32_t sK0 = sdO + Gm::Q_BYTES;
  const uint32_t sV0 = sK0 + ST * Gm::KV_BYTES;

  const int bh = blockIdx.x;
  const int b = bh / p.Hq, hq = bh - b * p.Hq;
  const int hk = hq / p.G;
  const int qt = p.n_qtiles - 1 - static_cast<int>(blockIdx.y);
  const int q0 = qt * BQ;
  const int q_hi = min(q0 + BQ, p.Lq);
  const int kv_end = CAUSAL ? min(p.Lk, q_hi + p.off) : p.Lk;
  const int n_kv = (kv_end + BK - 1) / BK;
  const WaitGuard g{&abort_flag, p.status, p.limit_ns};

  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(smem_u32(&bar_q), 1);
    for (int s = 0; s < ST; ++s) {
      mbar_init(smem_u32(&bar_kfull[s]), 1);
      mbar_init(smem_u32(&bar_vfull[s]), 1);
      mbar_init(smem_u32(&bar_kvempty[s]), 1);
    }
    mbar_init(smem_u32(&bar_sfull), 1);
    mbar_init(smem_u32(&bar_dsready), 128);
    mbar_init(smem_u32(&bar_dqdone), 1);
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
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      tma_prefetch_desc(&tmdO);
      const int zkv = b * p.Hkv + hk;
      mbar_arrive_expect_tx(smem_u32(&bar_q), 2 * Gm::Q_BYTES);
      for (int c = 0; c < NCH; ++c) {
        tma_load_3d(sQ + c * BQ * 128, &tmQ, smem_u32(&bar_q), c * 64, q0, bh);
        tma_load_3d(sdO + c * BQ * 128, &tmdO, smem_u32(&bar_q), c * 64, q0, bh);
      }
      for (int j = 0; j < n_kv; ++j) {
        const int s = j % ST, u = j / ST;
        if (u > 0) mbar_wait(smem_u32(&bar_kvempty[s]), (u - 1) & 1, g, kDevTimeoutBase + 11);
        mbar_arrive_expect_tx(smem_u32(&bar_kfull[s]), Gm::KV_BYTES);
        for (int c = 0; c < NCH; ++c)
          tma_load_3d(sK0 + s * Gm::KV_BYTES + c * BK * 128, &tmK, smem_u32(&bar_kfull[s]), c * 64,
                      j * BK, zkv);
        mbar_arrive_expect_tx(smem_u32(&bar_vfull[s]), Gm::KV_BYTES);
        for (int c = 0; c < NCH; ++c)
          tma_load_3d(sV0 + s * Gm::KV_BYTES + c * BK * 128, &tmV, smem_u32(&bar_vfull[s]), c * 64,
                      j * BK, zkv);
      }
      for (int j = (n_kv > ST ? n_kv - ST : 0); j < n_kv; ++j)
        mbar_wait_drain(smem_u32(&bar_vfull[j % ST]), (j / ST) & 1, p.limit_ns);
    }
  } else if (warp == 5) {
    if (lane == 0) {
      constexpr uint32_t IDESC_S = make_idesc_f16(128, BK, BF16, false, false);
      constexpr uint32_t IDESC_DQ = make_idesc_f16(128, D, BF16, false, true);
      mbar_wait(smem_u32(&bar_q), 0, g, kDevTimeoutBase + 12);
      tc_fence_after_sync();
      for (int j = 0; j < n_kv; ++j) {
        const int s = j % ST;
        const uint32_t kbase = sK0 + s * Gm::KV_BYTES, vbase = sV0 + s * Gm::KV_BYTES;
        mbar_wait(smem_u32(&bar_kfull[s]), (j / ST) & 1, g, kDevTimeoutBase + 13);
        tc_fence_after_sync();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t qo = (kk >> 2) * (BQ * 128) + (kk & 3) * 32;
          const uint32_t ko = (kk >> 2) * (BK * 128) + (kk & 3) * 32;
          mma_ss(tmem + Gm::S_COL, make_sdesc_sw128(sQ + qo, 16, 1024),
                 make_sdesc_sw128(kbase + ko, 16, 1024), IDESC_S, kk > 0 ? 1u : 0u);
        }
        mbar_wait(smem_u32(&bar_vfull[s]), (j / ST) & 1, g, kDevTimeoutBase + 14);
        tc_fence_after_sync();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t qo = (kk >> 2) * (BQ * 128) + (kk & 3) * 32;
          const uint32_t ko = (kk >> 2) * (BK * 128) + (kk & 3) * 32;
          mma_ss(tmem + Gm::DP_COL, make_sdesc_sw128(sdO + qo, 16, 1024),
                 make_sdesc_sw128(vbase + ko, 16, 1024), IDESC_S, kk > 0 ? 1u : 0u);
        }
        mma_commit(smem_u32(&bar_sfull));
        mbar_wait(smem_u32(&bar_dsready), j & 1, g, kDevTimeoutBase + 15);
        tc_fence_after_sync();
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk) {
          mma_ts(tmem + Gm::DQ_COL, tmem + Gm::DS_COL + kk * 8,
                 make_sdesc_sw128(kbase + kk * 2048, BK * 128, 1024), IDESC_DQ,
                 (j > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(smem_u32(&bar_kvempty[s]));
      }
      mma_commit(smem_u32(&bar_dqdone));
      mbar_wait_drain(smem_u32(&bar_dqdone), 0, p.limit_ns);
    }
  } else {
    const int r = warp * 32 + lane;
    const int qi = q0 + r;
    const uint32_t lrow = static_cast<uint32_t>(warp * 32) << 16;
    const float sl2 = p.scale_log2;
    const size_t row = static_cast<size_t>(bh) * p.Lq + qi;
    const float lse_r = qi < p.Lq ? p.lse[row] : 0.f;
    const float dlt_r = qi < p.Lq ? p.delta[row] : 0.f;
    const int lim = CAUSAL ? min(qi + p.off, p.Lk - 1) : p.Lk - 1;
    for (int j = 0; j < n_kv; ++j) {
      mbar_wait(smem_u32(&bar_sfull), j & 1, g, kDevTimeoutBase + 16);
      __syncwarp();
      tc_fence_after_sync();
      const int k0 = j * BK;
      const bool need_mask = (CAUSAL && (k0 + BK - 1 > q0 + p.off)) || (k0 + BK > p.Lk);
#pragma unroll
      for (int c = 0; c < BK / 32; ++c) {
        uint32_t sr[32], dr[32];
        tmem_ld32(tmem + lrow + Gm::S_COL + c * 32, sr);
        tmem_ld32(tmem + lrow + Gm::DP_COL + c * 32, dr);
        tmem_ld_wait(sr);
        reg_fence(dr);
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          float p0 = ex2_approx(fmaf(__uint_as_float(sr[2 * i]), sl2, -lse_r));
          float p1 = ex2_approx(fmaf(__uint_as_float(sr[2 * i + 1]), sl2, -lse_r));
          if (need_mask) {
            if (k0 + c * 32 + 2 * i > lim) p0 = 0.f;
            if (k0 + c * 32 + 2 * i + 1 > lim) p1 = 0.f;
          }
          const float ds0 = p0 * (__uint_as_float(dr[2 * i]) - dlt_r);
          const float ds1 = p1 * (__uint_as_float(dr[2 * i + 1]) - dlt_r);
          pk[i] = E::pack(ds0, ds1);
        }
        tmem_st16(tmem + lrow + Gm::DS_COL + c * 16, pk);
      }
      tmem_st_wait();
      tc_fence_before_sync();
      mbar_arrive(smem_u32(&bar_dsready));
    }
    mbar_wait(smem_u32(&bar_dqdone), 0, g, kDevTimeoutBase + 17);
    __syncwarp();
    tc_fence_after_sync();
    typename E::T* dqrow = reinterpret_cast<typename E::T*>(p.dq) + row * D;
#pragma unroll 1
    for (int c = 0; c < D / 32; ++c) {
      uint32_t rr[32];
      tmem_ld32(tmem + lrow + Gm::DQ_COL + c * 32, rr);
      tmem_ld_wait(rr);
      if (qi < p.Lq) store_row32<BF16>(dqrow + c * 32, rr, p.scale);
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
