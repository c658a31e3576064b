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
// Pipelining: S^T and dP^T are double-buffered in tensor memory, so the MMAs
// of query tile i+1 run while the row threads turn tile i into P^T and dS^T.
// P^T and dS^T (16-bit pairs) are written back over the fp32 S^T / dP^T
// columns the same warpgroup has just read, and the dV / dK MMAs read them
// from there.  The next MMA that writes those columns is issued after the
// MMAs that read them, by the same thread, and tcgen05 MMAs of one CTA run
// in issue order.
//
// MODE selects which outputs one CTA accumulates.  kDkvBoth keeps dK and dV
// in tensor memory together (D <= 128).  At D = 256 the two accumulators
// alone fill the 512 TMEM columns, so dV (kDkvDvOnly: S^T, P^T, dV) and dK
// (kDkvDkOnly: S^T, dP^T, dS^T, dK) are produced by separate CTAs of one
// launch (attn_bwd_dkv_kernel below).
//
// Warp roles (320 threads): warps 0-7 row threads -- warp w owns TMEM lanes
// 32*(w%4)..+31 (key rows) and query columns 32*(w/4)..+31 of each tile;
// warp 8 producer (TMA for Q/dO tiles, plain loads for the per-query
// lse/delta values); warp 9 MMA issuer and TMEM owner.  MMA issue competes
// with MUFU instructions issued on the same SM sub-partition, so the row warps
// on sub-partition 1 evaluate part of their exponentials with a polynomial on
// the FMA pipe (ex2_poly2).
#pragma once

#include <type_traits>

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
  static constexpr int ST_COL = (MODE == kDkvBoth) ? 2 * ACC_W : ACC_W;  // two buffers of BQ columns
  static constexpr int DPT_COL = ST_COL + 2 * BQ;                        // two buffers (not in DvOnly)
  static constexpr int TMEM_COLS = 512;
  static constexpr int NUM_COMPUTE_WARPS = 8;
  static constexpr int NUM_THREADS = 32 * (NUM_COMPUTE_WARPS + 2);
  static constexpr int PRODUCER_WARP = NUM_COMPUTE_WARPS;
  static constexpr int MMA_WARP = NUM_COMPUTE_WARPS + 1;
  static_assert(STAGES >= 1, "shared memory budget");
  // element pairs (of 16 per thread and query tile) whose exponentials use
  // the polynomial on the MMA warp's sub-partition
#ifndef GBATTN_DKV_POLY_PAIRS
  static constexpr int POLY_PAIRS = 10;
#else
  static constexpr int POLY_PAIRS = GBATTN_DKV_POLY_PAIRS;
#endif
  static_assert(POLY_PAIRS >= 0 && POLY_PAIRS <= 16, "polynomial share");
  static_assert(MODE != kDkvBoth || D <= 128, "dK and dV together need D <= 128");
  static_assert((NEED_DS ? DPT_COL + 2 * BQ : ST_COL + 2 * BQ) <= TMEM_COLS, "tensor memory budget");
};

// One CTA's work: key tile kt of KV head bhk = b * Hkv + hk, in mode MODE.
template <int D, bool BF16, bool CAUSAL, int MODE>
__device__ __forceinline__ void dkv_tile(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                                         const CUtensorMap& tmdO, const BwdParams& p, const int bhk, const int kt) {
  using Gm = DkvGeom<D, MODE>;
  using E = Elem<BF16>;
  constexpr int BQ = Gm::BQ, BK = Gm::BK, NCH = Gm::NCH, ST = Gm::STAGES;
  constexpr int NCT = 32 * Gm::NUM_COMPUTE_WARPS;  // row threads

  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t bar_kv, bar_stfull[ST], bar_stempty[ST], bar_sfull[2], bar_pready[2], bar_accdone;
  __shared__ __align__(16) float nlse_s[ST][BQ];  // -lse per query column
  __shared__ __align__(16) float dlt_s[ST][BQ];
  __shared__ uint32_t tmem_slot;
  __shared__ volatile int abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t sK = sbase;
  const uint32_t sV = sK + Gm::K_BYTES;  // only when NEED_V
  const uint32_t sQ0 = sbase + Gm::RES_BYTES;
  const uint32_t sdO0 = sQ0 + ST * Gm::Q_BYTES;

  const int b = bhk / p.Hkv, hk = bhk - b * p.Hkv;
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
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&bar_sfull[i]), 1);
      mbar_init(smem_u32(&bar_pready[i]), NCT);
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
  tc_fence_after_sync();
  const uint32_t tmem = tmem_slot;

  if (warp == Gm::PRODUCER_WARP) {
    // ---------------- producer (whole warp) ----------------
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmdO);
      if (Gm::NEED_V) tma_prefetch_desc(&tmV);
    }
    __syncwarp();
    mbar_arrive_expect_tx_w(smem_u32(&bar_kv), Gm::RES_BYTES);
    for (int c = 0; c < NCH; ++c) {
      tma_load_3d_w(sK + c * BK * 128, &tmK, smem_u32(&bar_kv), c * 64, k0, bhk);
      if (Gm::NEED_V) tma_load_3d_w(sV + c * BK * 128, &tmV, smem_u32(&bar_kv), c * 64, k0, bhk);
    }
    for (int it = 0; it < n_iter; ++it) {
      const int s = it % ST, u = it / ST;
      if (u > 0) mbar_wait(smem_u32(&bar_stempty[s]), (u - 1) & 1, g, kDevTimeoutBase + 21);
      __syncwarp();
      const int gi = it / nq;
      const int q0 = (qt_start + (it - gi * nq)) * BQ;
      const int zq = b * p.Hq + hk * p.G + gi;
      mbar_arrive_expect_tx_w(smem_u32(&bar_stfull[s]), 2 * Gm::Q_BYTES);
      for (int c = 0; c < NCH; ++c) {
        tma_load_3d_w(sQ0 + s * Gm::Q_BYTES + c * BQ * 128, &tmQ, smem_u32(&bar_stfull[s]), c * 64, q0, zq);
        tma_load_3d_w(sdO0 + s * Gm::Q_BYTES + c * BQ * 128, &tmdO, smem_u32(&bar_stfull[s]), c * 64, q0, zq);
      }
#pragma unroll
      for (int t = 0; t < BQ / 32; ++t) {
        const int c = lane + 32 * t;
        const int qi = q0 + c;
        const size_t row = static_cast<size_t>(zq) * p.Lq + qi;
        nlse_s[s][c] = qi < p.Lq ? -p.lse[row] : -INFINITY;
        dlt_s[s][c] = (Gm::NEED_DS && qi < p.Lq) ? p.delta[row] : 0.f;
      }
      mbar_arrive(smem_u32(&bar_stfull[s]));
    }
    for (int it = (n_iter > ST ? n_iter - ST : 0); it < n_iter; ++it)
      mbar_wait_drain(smem_u32(&bar_stfull[it % ST]), (it / ST) & 1, p.limit_ns);
  } else if (warp == Gm::MMA_WARP) {
    // ---------------- MMA issuer (whole warp, one elected lane issues) ----------------
    constexpr uint32_t IDESC_S = make_idesc_f16(128, BQ, BF16, false, false);
    constexpr uint32_t IDESC_ACC = make_idesc_f16(128, D, BF16, false, true);
    const uint64_t dK = make_sdesc_sw128(sK, 16, 1024);             // K tile, K-major
    const uint64_t dV = make_sdesc_sw128(sV, 16, 1024);             // V tile, K-major
    const uint64_t dQk = make_sdesc_sw128(sQ0, 16, 1024);           // Q stage 0, K-major
    const uint64_t dOk = make_sdesc_sw128(sdO0, 16, 1024);          // dO stage 0, K-major
    const uint64_t dQm = make_sdesc_sw128(sQ0, BQ * 128, 1024);     // Q stage 0, MN-major
    const uint64_t dOm = make_sdesc_sw128(sdO0, BQ * 128, 1024);    // dO stage 0, MN-major
    mbar_wait(smem_u32(&bar_kv), 0, g, kDevTimeoutBase + 22);
    __syncwarp();
    tc_fence_after_sync();
    // S^T (and dP^T) of iteration `it` into buffer it & 1
    auto issue_s = [&](int it) {
      const int s = it % ST, buf = it & 1;
      mbar_wait(smem_u32(&bar_stfull[s]), (it / ST) & 1, g, kDevTimeoutBase + 23);
      __syncwarp();
      tc_fence_after_sync();
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t ko = (kk >> 2) * (BK * 128) + (kk & 3) * 32;
        const uint32_t qo = s * Gm::Q_BYTES + (kk >> 2) * (BQ * 128) + (kk & 3) * 32;
        mma_ss_w(tmem + Gm::ST_COL + buf * BQ, sdesc_add(dK, ko), sdesc_add(dQk, qo), IDESC_S, kk > 0 ? 1u : 0u);
        if (Gm::NEED_DS)
          mma_ss_w(tmem + Gm::DPT_COL + buf * BQ, sdesc_add(dV, ko), sdesc_add(dOk, qo), IDESC_S,
                   kk > 0 ? 1u : 0u);
      }
      mma_commit_w(smem_u32(&bar_sfull[buf]));
    };
    // With a single Q/dO stage the next tile can only be loaded once this
    // tile's dV/dK MMAs are done, so the next S^T is issued after them.
    constexpr bool kAhead = ST >= 2;
    if (n_iter > 0) issue_s(0);
    for (int it = 0; it < n_iter; ++it) {
      if (kAhead && it + 1 < n_iter) issue_s(it + 1);
      const int s = it % ST, buf = it & 1;
      mbar_wait(smem_u32(&bar_pready[buf]), (it >> 1) & 1, g, kDevTimeoutBase + 24);
      __syncwarp();
      tc_fence_after_sync();
      // A operand: 16 queries per K step; queries 32w'..32w'+31 of warpgroup
      // w' sit as pairs in columns 32w'..32w'+15 of the buffer.
#pragma unroll
      for (int kk = 0; kk < BQ / 16; ++kk) {
        const uint32_t acol = buf * BQ + (kk >> 1) * 32 + (kk & 1) * 8;
        const uint32_t bo = s * Gm::Q_BYTES + kk * 2048;
        if (Gm::NEED_DV)
          mma_ts_w(tmem + Gm::DV_COL, tmem + Gm::ST_COL + acol, sdesc_add(dOm, bo), IDESC_ACC,
                   (it > 0 || kk > 0) ? 1u : 0u);
        if (Gm::NEED_DS)
          mma_ts_w(tmem + Gm::DK_COL, tmem + Gm::DPT_COL + acol, sdesc_add(dQm, bo), IDESC_ACC,
                   (it > 0 || kk > 0) ? 1u : 0u);
      }
      mma_commit_w(smem_u32(&bar_stempty[s]));
      if (!kAhead && it + 1 < n_iter) issue_s(it + 1);
    }
    mma_commit_w(smem_u32(&bar_accdone));
    mbar_wait_drain(smem_u32(&bar_accdone), 0, p.limit_ns);
    __syncwarp();
  } else {
    // ---------------- key-row threads ----------------
    const int quad = warp & 3;        // TMEM lane quadrant
    const int half = warp >> 2;       // query columns 32*half .. +31
    const int r = quad * 32 + lane;
    const int kj = k0 + r;
    const uint32_t lrow = static_cast<uint32_t>(quad * 32) << 16;
    const float sl2 = p.scale_log2;
    const uint64_t sl2x2 = f2_pack(sl2, sl2);
    const int qmin = kj - p.off;  // causal: queries below this index cannot see key kj
    for (int it = 0; it < n_iter; ++it) {
      const int s = it % ST, buf = it & 1;
      const int gi = it / nq;
      const int q0 = (qt_start + (it - gi * nq)) * BQ;
      mbar_wait(smem_u32(&bar_stfull[s]), (it / ST) & 1, g, kDevTimeoutBase + 25);
      mbar_wait(smem_u32(&bar_sfull[buf]), (it >> 1) & 1, g, kDevTimeoutBase + 26);
      __syncwarp();
      tc_fence_after_sync();
      const bool need_mask = CAUSAL && (q0 < k0 + BK - 1 - p.off);
      const uint32_t scol = tmem + lrow + Gm::ST_COL + buf * BQ + half * 32;
      const uint32_t dcol = tmem + lrow + Gm::DPT_COL + buf * BQ + half * 32;
      uint32_t sr[32], dr[32];
      tmem_ld32(scol, sr);
      if (Gm::NEED_DS) tmem_ld32(dcol, dr);
      tmem_ld_wait(sr);
      if (Gm::NEED_DS) reg_fence(dr);
      const uint64_t* nlse_row = reinterpret_cast<const uint64_t*>(&nlse_s[s][half * 32]);
      const uint64_t* dlt_row = reinterpret_cast<const uint64_t*>(&dlt_s[s][half * 32]);
      const int qc0 = q0 + half * 32;
      uint32_t pk[16], dk[16];
      // NPOLY of the 16 pairs, spread evenly, use the polynomial
      auto pds_tile = [&](auto npoly_tag) {
        constexpr int NPOLY = decltype(npoly_tag)::value;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int c0 = 2 * i;
          float x0, x1, p0, p1;
          f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[c0]), __uint_as_float(sr[c0 + 1])), sl2x2, nlse_row[i]), x0, x1);
          if ((i + 1) * NPOLY / 16 > i * NPOLY / 16) {
            ex2_poly2(x0, x1, p0, p1);
          } else {
            p0 = ex2_approx(x0);
            p1 = ex2_approx(x1);
          }
          if (need_mask) {
            if (qc0 + c0 < qmin) p0 = 0.f;
            if (qc0 + c0 + 1 < qmin) p1 = 0.f;
          }
          pk[i] = E::pack(p0, p1);
          if (Gm::NEED_DS) {
            const uint64_t d2 = f2_sub(f2_pack(__uint_as_float(dr[c0]), __uint_as_float(dr[c0 + 1])), dlt_row[i]);
            float ds0, ds1;
            f2_unpack(f2_mul(f2_pack(p0, p1), d2), ds0, ds1);
            dk[i] = E::pack(ds0, ds1);
          }
        }
      };
      if (quad == 1)  // sub-partition of the MMA warp
        pds_tile(std::integral_constant<int, Gm::POLY_PAIRS>{});
      else
        pds_tile(std::integral_constant<int, 0>{});
      if (Gm::NEED_DV) tmem_st16(scol, pk);
      if (Gm::NEED_DS) tmem_st16(dcol, dk);
      tmem_st_wait();
      tc_fence_before_sync();
      mbar_arrive(smem_u32(&bar_pready[buf]));
    }
    mbar_wait(smem_u32(&bar_accdone), 0, g, kDevTimeoutBase + 27);
    __syncwarp();
    tc_fence_after_sync();
    // epilogue: warpgroup `half` writes output columns [half*D/2, (half+1)*D/2)
    const size_t row = static_cast<size_t>(bhk) * p.Lk + kj;
    if (Gm::NEED_DS) {
      typename E::T* dst = reinterpret_cast<typename E::T*>(p.dk) + row * D;
#pragma unroll 1
      for (int c = half; c < D / 32; c += 2) {
        uint32_t rr[32];
        tmem_ld32(tmem + lrow + Gm::DK_COL + c * 32, rr);
        tmem_ld_wait(rr);
        if (kj < p.Lk) store_row32<BF16>(dst + c * 32, rr, p.scale);
      }
    }
    if (Gm::NEED_DV) {
      typename E::T* dst = reinterpret_cast<typename E::T*>(p.dv) + row * D;
#pragma unroll 1
      for (int c = half; c < D / 32; c += 2) {
        uint32_t rr[32];
        tmem_ld32(tmem + lrow + Gm::DV_COL + c * 32, rr);
        tmem_ld_wait(rr);
        if (kj < p.Lk) store_row32<BF16>(dst + c * 32, rr, 1.f);
      }
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == Gm::MMA_WARP) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, Gm::TMEM_COLS);
  }
}

// D = 256: both halves in one launch, x = 2 * (b * Hkv + hk) + (0: dV, 1: dK),
// y = key tile.  CTAs are dispatched in x-then-y order, so the heavy key tiles
// (small kt: the most visible query tiles under causal masking) of both halves
// start first and the light ones of either half fill the tail.
template <int D>
struct DkvPairGeom {
  using Dv = DkvGeom<D, kDkvDvOnly>;
  using Dk = DkvGeom<D, kDkvDkOnly>;
  static_assert(Dv::NUM_THREADS == Dk::NUM_THREADS, "one block size for both halves");
  static constexpr int NUM_THREADS = Dv::NUM_THREADS;
  static constexpr int SMEM_BYTES = Dv::SMEM_BYTES > Dk::SMEM_BYTES ? Dv::SMEM_BYTES : Dk::SMEM_BYTES;
  static constexpr int BQ = Dv::BQ, BK = Dv::BK;
};

template <int D, bool BF16, bool CAUSAL>
__global__ void __launch_bounds__(DkvPairGeom<D>::NUM_THREADS, 1)
    attn_bwd_dkv_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                        const BwdParams p) {
  const int bhk = static_cast<int>(blockIdx.x >> 1), kt = static_cast<int>(blockIdx.y);
  if (blockIdx.x & 1)
    dkv_tile<D, BF16, CAUSAL, kDkvDkOnly>(tmQ, tmK, tmV, tmdO, p, bhk, kt);
  else
    dkv_tile<D, BF16, CAUSAL, kDkvDvOnly>(tmQ, tmK, tmV, tmdO, p, bhk, kt);
}

}  // namespace gbattn
