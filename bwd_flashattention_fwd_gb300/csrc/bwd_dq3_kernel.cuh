// Backward, dQ kernel for head dims up to 128: same mathematics as
// bwd_dq_kernel.cuh ("feat(attention): complete Flash Attention VJP
// implementation", sections "Background" and "Two-Kernel Design": the dQ
// kernel owns query rows and loops over key tiles; S = Q K^T and dP = dO V^T
// are recomputed, P = exp2(S * scale_log2 - lse), dS = P * (dP - delta),
// dQ += dS K, and dQ is scaled by `scale` at the end).
//
// Shared-memory bandwidth (128 B per clock per SM) is what limits an MMA
// whose two operands both come from shared memory at N = 64.  Q and dO do not
// change over the CTA's key loop, so the row threads copy them once into
// tensor memory and every MMA reads its A operand from there: S = Q K^T and
// dP = dO V^T read only the K / V tile from shared memory, dQ += dS K reads dS
// from tensor memory.  Tensor memory (512 columns): dQ (D), Q and dO (D/2
// columns of 16-bit pairs each), one S buffer and three dP buffers of 64
// columns; dS (16-bit pairs) is written back over the dP columns its warp
// has read.  Two warps issue the MMAs, each in an order that needs no
// completion round trip (tcgen05 MMAs of one issuing thread execute in issue
// order):
//   * the S warp issues S(j+1) as soon as every row thread has loaded S(j)
//     into registers ("S free" barrier), so it runs while the rows compute;
//   * the dQ warp issues dQ(j) += dS(j) K_j and then dP(j+3) into dP buffer
//     j mod 3, behind the MMA that reads dS(j) from it; three buffers keep
//     dP two tiles ahead of the row threads.
//
// Warp roles (352 threads): warps 0-7 row threads -- warp w owns TMEM lanes
// 32*(w%4)..+31 (query rows) and key columns 32*(w/4)..+31 of each 64-key
// tile, and copies D/2 columns of its rows of Q and dO into tensor memory;
// warp 8 TMA producer (K_j and V_j together into one ring stage); warp 9
// issues S = Q K^T and owns the TMEM allocation; warp 10 issues dQ += dS K
// and dP = dO V^T.
// MMA issue competes with MUFU instructions issued on the same SM
// sub-partition, so the row warps on sub-partitions 1 and 2 evaluate part of
// their exponentials with a polynomial on the FMA pipe (ex2_poly2).
#pragma once

#include <type_traits>

#include "kernel_common.cuh"

namespace gbattn {

template <int D>
struct Dq3Geom {
  static constexpr int BQ = 128;
  static constexpr int BK = 64;
  static constexpr int NCH = n_chunks(D);
  static constexpr int KV_BYTES = NCH * BK * 128;
  static constexpr int AVAIL = kMaxDynSmem - 512 - 1024;
  static constexpr int STAGES = AVAIL / (2 * KV_BYTES) > 6 ? 6 : AVAIL / (2 * KV_BYTES);  // K_j + V_j each
  static constexpr int SMEM_BYTES = 1024 + STAGES * 2 * KV_BYTES;
  static constexpr int DQ_COL = 0, Q_COL = 128, DO_COL = 192, S_COL = 256, DP_COL = 320;  // dP: 3 x 64
  static constexpr int NDP = 3;  // dP buffers
  static constexpr int TMEM_COLS = 512;
#ifndef GBATTN_DQ_ROW_WARPS
  static constexpr int NUM_COMPUTE_WARPS = 8;
#else
  static constexpr int NUM_COMPUTE_WARPS = GBATTN_DQ_ROW_WARPS;
#endif
  static constexpr int NG = NUM_COMPUTE_WARPS / 4;  // row warps per TMEM lane quadrant
  static constexpr int KC = BK / NG;                 // key columns per row warp
  static_assert(NUM_COMPUTE_WARPS == 8 || NUM_COMPUTE_WARPS == 16, "row warps");
  static constexpr int NCT = 32 * NUM_COMPUTE_WARPS;
  static constexpr int PRODUCER_WARP = NUM_COMPUTE_WARPS;
  static constexpr int S_MMA_WARP = NUM_COMPUTE_WARPS + 1;
  static constexpr int DQ_MMA_WARP = NUM_COMPUTE_WARPS + 2;
  static constexpr int NUM_THREADS = 32 * (NUM_COMPUTE_WARPS + 3);
  static_assert(D <= 128, "dQ, Q, dO and the S / dP buffers fill TMEM at D = 128");
  static_assert(STAGES >= NDP + 1, "dP of tile j+3 is issued while K_j is still in use");
  // element pairs (of 16 per thread and key tile) whose exponentials use the
  // polynomial, on the sub-partition of the S warp (1) and of the dQ / dP
  // warp (2)
#ifndef GBATTN_DQ_POLY_Q1
  static constexpr int POLY_Q1 = 0;
#else
  static constexpr int POLY_Q1 = GBATTN_DQ_POLY_Q1;
#endif
#ifndef GBATTN_DQ_POLY_Q2
  static constexpr int POLY_Q2 = 8;
#else
  static constexpr int POLY_Q2 = GBATTN_DQ_POLY_Q2;
#endif
  static_assert(POLY_Q1 >= 0 && POLY_Q1 <= 16 && POLY_Q2 >= 0 && POLY_Q2 <= 16, "polynomial share");
};

template <int D, bool BF16, bool CAUSAL>
__global__ void __launch_bounds__(Dq3Geom<D>::NUM_THREADS, 1)
    attn_bwd_dq3_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                        const void* __restrict__ q, const void* __restrict__ dO, const BwdParams p) {
  using Gm = Dq3Geom<D>;
  using E = Elem<BF16>;
  constexpr int BQ = Gm::BQ, BK = Gm::BK, NCH = Gm::NCH, ST = Gm::STAGES;

  extern __shared__ uint8_t smem_raw[];
  constexpr int NDP = Gm::NDP;
  __shared__ uint64_t bar_qready, bar_kvfull[ST], bar_kvempty[ST], bar_sfull, bar_sfree, bar_dpfull[NDP],
      bar_dsready[NDP], bar_dqdone;
  __shared__ uint32_t tmem_slot;
  __shared__ volatile int abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t sK0 = sbase;  // stage s: K at sK0 + 2s * KV_BYTES, V right after

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
    mbar_init(smem_u32(&bar_qready), Gm::NCT);
    for (int s = 0; s < ST; ++s) {
      mbar_init(smem_u32(&bar_kvfull[s]), 1);
      mbar_init(smem_u32(&bar_kvempty[s]), 2);  // S (S warp) and dP, dQ (dQ warp) read the stage
    }
    mbar_init(smem_u32(&bar_sfull), 1);
    mbar_init(smem_u32(&bar_sfree), Gm::NCT);
    for (int i = 0; i < NDP; ++i) {
      mbar_init(smem_u32(&bar_dpfull[i]), 1);
      mbar_init(smem_u32(&bar_dsready[i]), Gm::NCT);
    }
    mbar_init(smem_u32(&bar_dqdone), 1);
    fence_mbar_init();
  }
  if (warp == Gm::S_MMA_WARP) {
    tmem_alloc(smem_u32(&tmem_slot), Gm::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = tmem_slot;

  if (warp == Gm::PRODUCER_WARP) {
    // ---------------- TMA producer (whole warp, one elected lane issues) ----------------
    if (lane == 0) {
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
    }
    __syncwarp();
    const int zkv = b * p.Hkv + hk;
    for (int j = 0; j < n_kv; ++j) {
      const int s = j % ST;
      if (j >= ST) mbar_wait(smem_u32(&bar_kvempty[s]), (j / ST - 1) & 1, g, kDevTimeoutBase + 61);
      __syncwarp();
      const uint32_t bar = smem_u32(&bar_kvfull[s]);
      const uint32_t dK = sK0 + 2 * s * Gm::KV_BYTES;
      mbar_arrive_expect_tx_w(bar, 2 * Gm::KV_BYTES);
      for (int c = 0; c < NCH; ++c) {
        tma_load_3d_w(dK + c * BK * 128, &tmK, bar, c * 64, j * BK, zkv);
        tma_load_3d_w(dK + Gm::KV_BYTES + c * BK * 128, &tmV, bar, c * 64, j * BK, zkv);
      }
    }
    for (int j = (n_kv > ST ? n_kv - ST : 0); j < n_kv; ++j)
      mbar_wait_drain(smem_u32(&bar_kvfull[j % ST]), (j / ST) & 1, p.limit_ns);
    __syncwarp();
  } else if (warp == Gm::S_MMA_WARP) {
    // ---------------- S = Q K^T issuer (A operand Q from tensor memory) ----------------
    constexpr uint32_t IDESC_S = make_idesc_f16(128, BK, BF16, false, false);
    const uint64_t dKk = make_sdesc_sw128(sK0, 16, 1024);  // K stage 0, K-major
    mbar_wait(smem_u32(&bar_qready), 0, g, kDevTimeoutBase + 63);
    __syncwarp();
    tc_fence_after_sync();
    for (int j = 0; j < n_kv; ++j) {
      const int s = j % ST;
      // every row thread has loaded S(j-1) from the buffer
      if (j >= 1) mbar_wait(smem_u32(&bar_sfree), (j - 1) & 1, g, kDevTimeoutBase + 64);
      mbar_wait(smem_u32(&bar_kvfull[s]), (j / ST) & 1, g, kDevTimeoutBase + 65);
      __syncwarp();
      tc_fence_after_sync();
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t ko = 2 * s * Gm::KV_BYTES + (kk >> 2) * (BK * 128) + (kk & 3) * 32;
        mma_ts_w(tmem + Gm::S_COL, tmem + Gm::Q_COL + kk * 8, sdesc_add(dKk, ko), IDESC_S, kk > 0 ? 1u : 0u);
      }
      mma_commit_w(smem_u32(&bar_sfull));
      mma_commit_w(smem_u32(&bar_kvempty[s]));
    }
    __syncwarp();
  } else if (warp == Gm::DQ_MMA_WARP) {
    // ---------------- dQ += dS K and dP = dO V^T issuer ----------------
    constexpr uint32_t IDESC_S = make_idesc_f16(128, BK, BF16, false, false);
    constexpr uint32_t IDESC_DQ = make_idesc_f16(128, D, BF16, false, true);
    const uint64_t dVk = make_sdesc_sw128(sK0 + Gm::KV_BYTES, 16, 1024);  // V stage 0, K-major
    const uint64_t dKm = make_sdesc_sw128(sK0, BK * 128, 1024);           // K stage 0, MN-major
    mbar_wait(smem_u32(&bar_qready), 0, g, kDevTimeoutBase + 66);
    __syncwarp();
    tc_fence_after_sync();
    auto issue_dp = [&](int j) {
      const int s = j % ST, buf = j % NDP;
      mbar_wait(smem_u32(&bar_kvfull[s]), (j / ST) & 1, g, kDevTimeoutBase + 67);
      __syncwarp();
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t vo = 2 * s * Gm::KV_BYTES + (kk >> 2) * (BK * 128) + (kk & 3) * 32;
        mma_ts_w(tmem + Gm::DP_COL + buf * BK, tmem + Gm::DO_COL + kk * 8, sdesc_add(dVk, vo), IDESC_S,
                 kk > 0 ? 1u : 0u);
      }
      mma_commit_w(smem_u32(&bar_dpfull[buf]));
    };
    for (int j = 0; j < NDP && j < n_kv; ++j) issue_dp(j);
    for (int j = 0; j < n_kv; ++j) {
      const int s = j % ST, buf = j % NDP;
      mbar_wait(smem_u32(&bar_dsready[buf]), (j / NDP) & 1, g, kDevTimeoutBase + 68);
      __syncwarp();
      tc_fence_after_sync();
      // A operand: 16 keys per K step; keys KC*h..KC*h+KC-1 of row-warp
      // group h sit as pairs in columns KC*h..KC*h+KC/2-1 of the dP buffer.
#pragma unroll
      for (int kk = 0; kk < BK / 16; ++kk) {
        const uint32_t acol = Gm::DP_COL + buf * BK + (16 * kk / Gm::KC) * Gm::KC + (16 * kk % Gm::KC) / 2;
        mma_ts_w(tmem + Gm::DQ_COL, tmem + acol, sdesc_add(dKm, 2 * s * Gm::KV_BYTES + kk * 2048), IDESC_DQ,
                 (j > 0 || kk > 0) ? 1u : 0u);
      }
      // this warp's dP(j) and dQ(j) are its last reads of the stage
      mma_commit_w(smem_u32(&bar_kvempty[s]));
      // dP(j+3) overwrites the buffer behind dQ(j), which reads its dS
      if (j + NDP < n_kv) issue_dp(j + NDP);
    }
    // Every S MMA completed before the last dS was ready, so this commit
    // covers all MMAs of the CTA.
    mma_commit_w(smem_u32(&bar_dqdone));
    mbar_wait_drain(smem_u32(&bar_dqdone), 0, p.limit_ns);
    __syncwarp();
  } else {
    // ---------------- row threads ----------------
    constexpr int NG = Gm::NG, KC = Gm::KC;
    const int quad = warp & 3;  // TMEM lane quadrant (query rows)
    const int grp = warp >> 2;  // key columns KC*grp .. +KC-1 of each tile
    const int r = quad * 32 + lane;
    const int qi = q0 + r;
    const uint32_t lrow = static_cast<uint32_t>(quad * 32) << 16;
    const float sl2 = p.scale_log2;
    const size_t row = static_cast<size_t>(bh) * p.Lq + qi;
    // Q and dO rows into tensor memory: this warp copies columns
    // [grp*D/NG, (grp+1)*D/NG) of its 32 rows (zeros past Lq), as 16-bit pairs.
    {
      constexpr int EW = D / NG;   // elements per thread per tensor
      constexpr int NV = EW / 8;   // 16-byte loads per thread per tensor
      constexpr int PC = EW / 2;   // packed columns per thread per tensor
      const uint4* qrow =
          reinterpret_cast<const uint4*>(reinterpret_cast<const typename E::T*>(q) + row * D + grp * EW);
      const uint4* orow =
          reinterpret_cast<const uint4*>(reinterpret_cast<const typename E::T*>(dO) + row * D + grp * EW);
      uint32_t qa[PC], oa[PC];
#pragma unroll
      for (int v = 0; v < NV; ++v) {
        uint4 x = make_uint4(0u, 0u, 0u, 0u), y = make_uint4(0u, 0u, 0u, 0u);
        if (qi < p.Lq) {
          x = qrow[v];
          y = orow[v];
        }
        qa[4 * v + 0] = x.x, qa[4 * v + 1] = x.y, qa[4 * v + 2] = x.z, qa[4 * v + 3] = x.w;
        oa[4 * v + 0] = y.x, oa[4 * v + 1] = y.y, oa[4 * v + 2] = y.z, oa[4 * v + 3] = y.w;
      }
      const uint32_t qcol = tmem + lrow + Gm::Q_COL + grp * PC, ocol = tmem + lrow + Gm::DO_COL + grp * PC;
      // PC packed columns (4 .. 32) in pieces of 16, 8 and 4
#pragma unroll
      for (int c = 0; c + 16 <= PC; c += 16) {
        uint32_t t[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) t[i] = qa[c + i];
        tmem_st16(qcol + c, t);
#pragma unroll
        for (int i = 0; i < 16; ++i) t[i] = oa[c + i];
        tmem_st16(ocol + c, t);
      }
      if constexpr (PC % 16 >= 8) {
        constexpr int c = PC / 16 * 16;
        uint32_t t[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) t[i] = qa[c + i];
        tmem_st8(qcol + c, t);
#pragma unroll
        for (int i = 0; i < 8; ++i) t[i] = oa[c + i];
        tmem_st8(ocol + c, t);
      }
      if constexpr (PC % 8 == 4) {
        constexpr int c = PC / 8 * 8;
        uint32_t t[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) t[i] = qa[c + i];
        tmem_st4(qcol + c, t);
#pragma unroll
        for (int i = 0; i < 4; ++i) t[i] = oa[c + i];
        tmem_st4(ocol + c, t);
      }
      tmem_st_wait();
      tc_fence_before_sync();
      mbar_arrive(smem_u32(&bar_qready));
    }
    const float lse_r = qi < p.Lq ? p.lse[row] : 0.f;
    const float dlt_r = qi < p.Lq ? p.delta[row] : 0.f;
    const uint64_t sl2x2 = f2_pack(sl2, sl2), nlse2 = f2_pack(-lse_r, -lse_r), dlt2 = f2_pack(dlt_r, dlt_r);
    const int lim = CAUSAL ? min(qi + p.off, p.Lk - 1) : p.Lk - 1;
    for (int j = 0; j < n_kv; ++j) {
      const int buf = j % NDP;
      mbar_wait(smem_u32(&bar_sfull), j & 1, g, kDevTimeoutBase + 69);
      mbar_wait(smem_u32(&bar_dpfull[buf]), (j / NDP) & 1, g, kDevTimeoutBase + 71);
      __syncwarp();
      tc_fence_after_sync();
      const int kc0 = j * BK + grp * KC;  // first key of this thread's columns
      const bool need_mask = (CAUSAL && (j * BK + BK - 1 > q0 + p.off)) || (j * BK + BK > p.Lk);
      const uint32_t dcol = tmem + lrow + Gm::DP_COL + buf * BK + grp * KC;
      uint32_t sr[KC], dr[KC];
      if constexpr (KC == 32) {
        tmem_ld32(tmem + lrow + Gm::S_COL + grp * KC, sr);
        tmem_ld32(dcol, dr);
      } else {
        tmem_ld16(tmem + lrow + Gm::S_COL + grp * KC, sr);
        tmem_ld16(dcol, dr);
      }
      tmem_ld_wait(sr);
      reg_fence(dr);
      // S(j) is in registers: the S warp may overwrite the buffer
      tc_fence_before_sync();
      mbar_arrive(smem_u32(&bar_sfree));
      uint32_t pk[KC / 2];
      // NPOLY of the KC/2 pairs, spread evenly, use the polynomial
      auto ds_tile = [&](auto npoly_tag) {
        constexpr int NPOLY = decltype(npoly_tag)::value * KC / 32;
#pragma unroll
        for (int i = 0; i < KC / 2; ++i) {
          float x0, x1, p0, p1;
          f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[2 * i]), __uint_as_float(sr[2 * i + 1])), sl2x2, nlse2), x0, x1);
          if ((i + 1) * NPOLY / (KC / 2) > i * NPOLY / (KC / 2)) {
            ex2_poly2(x0, x1, p0, p1);
          } else {
            p0 = ex2_approx(x0);
            p1 = ex2_approx(x1);
          }
          if (need_mask) {
            if (kc0 + 2 * i > lim) p0 = 0.f;
            if (kc0 + 2 * i + 1 > lim) p1 = 0.f;
          }
          const uint64_t d2 = f2_sub(f2_pack(__uint_as_float(dr[2 * i]), __uint_as_float(dr[2 * i + 1])), dlt2);
          float ds0, ds1;
          f2_unpack(f2_mul(f2_pack(p0, p1), d2), ds0, ds1);
          pk[i] = E::pack(ds0, ds1);
        }
      };
      if (quad == 1)  // sub-partition of the S warp
        ds_tile(std::integral_constant<int, Gm::POLY_Q1>{});
      else if (quad == 2)  // sub-partition of the dQ / dP warp
        ds_tile(std::integral_constant<int, Gm::POLY_Q2>{});
      else
        ds_tile(std::integral_constant<int, 0>{});
      if constexpr (KC == 32)
        tmem_st16(dcol, pk);
      else
        tmem_st8(dcol, pk);
      tmem_st_wait();
      tc_fence_before_sync();
      mbar_arrive(smem_u32(&bar_dsready[buf]));
    }
    mbar_wait(smem_u32(&bar_dqdone), 0, g, kDevTimeoutBase + 70);
    __syncwarp();
    tc_fence_after_sync();
    typename E::T* dqrow = reinterpret_cast<typename E::T*>(p.dq) + row * D;
#pragma unroll 1
    for (int c = grp; c < D / 32; c += NG) {
      uint32_t rr[32];
      tmem_ld32(tmem + lrow + Gm::DQ_COL + c * 32, rr);
      tmem_ld_wait(rr);
      if (qi < p.Lq) store_row32<BF16>(dqrow + c * 32, rr, p.scale);
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == Gm::S_MMA_WARP) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, Gm::TMEM_COLS);
  }
}

}  // namespace gbattn
