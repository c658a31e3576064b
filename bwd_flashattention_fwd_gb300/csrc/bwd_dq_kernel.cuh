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
// Pipelining: S and dP are double-buffered in tensor memory (key tiles of
// BK = 64), so the MMAs of key tile j+1 run while the row threads turn tile j
// into dS.  dS (16-bit pairs) is written back over the fp32 S columns the same
// warpgroup has just read, and the dQ MMA reads it from there.  Two warps issue
// the MMAs: one S / dP, one dQ += dS K (a single issuing warp spends more time
// in barrier waits and commits than the tensor core needs for a tile).  MMAs of
// different issuing threads are not ordered, so the S warp waits on a "buffer
// free" barrier, committed after the dQ MMA that read the buffer, before it
// writes that buffer again.  K and V tiles arrive in separate TMA rings: V is
// released as soon as dP has used it, K only after dQ += dS K.
//
// Warp roles (352 threads): warps 0-7 row threads -- warp w owns TMEM lanes
// 32*(w%4)..+31 (query rows) and key columns 32*(w/4)..+31 of each tile;
// warp 8 TMA producer; warp 9 issues S / dP and owns the TMEM allocation;
// warp 10 issues dQ += dS K.
//
// DECODE (short query lengths): as in the forward kernel, one packed tile
// holds the G query heads x Lq rows of a KV head (row r is query r % Lq) and
// CTA (x, y) covers key tiles [y*split_tiles, ...); it writes its fp32 share
// of dS K per row, and a reduction kernel sums the shares and applies the
// scale.  P uses the final lse, so the shares simply add.
//
// MASKED: block-sparse variant ("feat(attention): complete Flash Attention
// VJP implementation", section "Sparse Block Masks": the dQ kernel skips the
// key blocks whose mask entry is zero); a query tile with no kept key block
// writes dQ = 0.
#pragma once

#include "kernel_common.cuh"

namespace gbattn {

template <int D>
struct DqGeom {
  static constexpr int BQ = 128;
  static constexpr int BK = 64;
  static constexpr int NCH = n_chunks(D);
  static constexpr int Q_BYTES = NCH * BQ * 128;
  static constexpr int KV_BYTES = NCH * BK * 128;
  // static shared memory here is only the barriers (< 512 B)
  static constexpr int AVAIL = kMaxDynSmem - 512 - 1024 - 2 * Q_BYTES;
  // K stays in flight longer (until dQ += dS K), so it gets the extra stage.
  static constexpr int KSTAGES = (AVAIL / KV_BYTES) >= 8 ? 4 : (AVAIL / KV_BYTES + 1) / 2;
  static constexpr int VSTAGES = (AVAIL / KV_BYTES - KSTAGES) > 4 ? 4 : (AVAIL / KV_BYTES - KSTAGES);
  static constexpr int SMEM_BYTES = 1024 + 2 * Q_BYTES + (KSTAGES + VSTAGES) * KV_BYTES;
  static constexpr int DQ_COL = 0;
  static constexpr int S_COL = (D <= 128) ? 128 : 256;  // two buffers of BK columns
  static constexpr int DP_COL = S_COL + 2 * BK;         // two buffers of BK columns
  static constexpr int TMEM_COLS = 512;
  static constexpr int NUM_COMPUTE_WARPS = 8;
  static constexpr int NUM_THREADS = 32 * (NUM_COMPUTE_WARPS + 3);
  static constexpr int ACC_MMA_WARP = NUM_COMPUTE_WARPS + 2;
  static constexpr int PRODUCER_WARP = NUM_COMPUTE_WARPS;
  static constexpr int MMA_WARP = NUM_COMPUTE_WARPS + 1;
  // S of tile j+1 is issued before dQ of tile j releases K_j: K needs 2 stages.
  static_assert(KSTAGES >= 2 && VSTAGES >= 1, "shared memory budget");
  static_assert(DP_COL + 2 * BK <= TMEM_COLS, "tensor memory budget");
};

template <int D, bool BF16, bool CAUSAL, bool DECODE = false, bool MASKED = false>
__global__ void __launch_bounds__(DqGeom<D>::NUM_THREADS, 1)
    attn_bwd_dq_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                       const BwdParams p) {
  using Gm = DqGeom<D>;
  using E = Elem<BF16>;
  constexpr int BQ = Gm::BQ, BK = Gm::BK, NCH = Gm::NCH, KST = Gm::KSTAGES, VST = Gm::VSTAGES;
  constexpr int NCT = 32 * Gm::NUM_COMPUTE_WARPS;

  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t bar_q, bar_kfull[KST], bar_kempty[KST], bar_vfull[VST], bar_vempty[VST], bar_sfull[2],
      bar_dsready[2], bar_pfree[2], bar_dqdone, bar_sdone;
  __shared__ uint32_t tmem_slot;
  __shared__ volatile int abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t sQ = sbase;
  const uint32_t sdO = sQ + Gm::Q_BYTES;
  const uint32_t sK0 = sdO + Gm::Q_BYTES;
  const uint32_t sV0 = sK0 + KST * Gm::KV_BYTES;

  const int bh = blockIdx.x;
  const int b = bh / p.Hq, hq = bh - b * p.Hq;
  const int hk = hq / p.G;
  const int qt = DECODE ? 0 : p.n_qtiles - 1 - static_cast<int>(blockIdx.y);
  const int q0 = qt * BQ;
  const int q_hi = min(q0 + BQ, p.Lq);
  const int kv_end = CAUSAL ? min(p.Lk, q_hi + p.off) : p.Lk;
  // key tiles [j0, j0 + n_kv) of this CTA
  const int j0 = DECODE ? static_cast<int>(blockIdx.y) * p.split_tiles : 0;
  const int n_kv = DECODE ? min((kv_end + BK - 1) / BK - j0, p.split_tiles) : (kv_end + BK - 1) / BK;
  static_assert(!(MASKED && DECODE), "no block mask on the decode path");
  static_assert(BQ == kMaskBlock && kMaskBlock % BK == 0, "query tile = mask block");
  // key tile jt is computed (block mask), and the number of computed tiles (warp-collective)
  auto keep = [&](int jt) { return !MASKED || mask_keep(p, qt, jt * BK / kMaskBlock); };
  const int nk = count_kept<MASKED>(keep, 0, n_kv);
  const WaitGuard g{&abort_flag, p.status, p.limit_ns};
  // extents for the debug build's index checks: rows of q / dq / lse /
  // delta, of dk / dv, and of the k / v buffers (pitch kv_pitch per head)
  [[maybe_unused]] const size_t n_qrows = static_cast<size_t>(p.B) * p.Hq * p.Lq;
  [[maybe_unused]] const size_t n_krows = static_cast<size_t>(p.B) * p.Hkv * p.Lk;
  [[maybe_unused]] const size_t n_kvbuf = (static_cast<size_t>(p.B) * p.Hkv - 1) * p.kv_pitch + p.Lk;

  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(smem_u32(&bar_q), 1);
    for (int s = 0; s < KST; ++s) {
      mbar_init(smem_u32(&bar_kfull[s]), 1);
      mbar_init(smem_u32(&bar_kempty[s]), 2);  // S (S warp) and dQ (dQ warp) read K_j
    }
    for (int s = 0; s < VST; ++s) {
      mbar_init(smem_u32(&bar_vfull[s]), 1);
      mbar_init(smem_u32(&bar_vempty[s]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&bar_sfull[i]), 1);
      mbar_init(smem_u32(&bar_dsready[i]), NCT);
      mbar_init(smem_u32(&bar_pfree[i]), 1);
    }
    mbar_init(smem_u32(&bar_dqdone), 1);
    mbar_init(smem_u32(&bar_sdone), 1);
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
    // ---------------- TMA producer (whole warp, one elected lane issues) ----------------
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      tma_prefetch_desc(&tmdO);
    }
    __syncwarp();
    const int zkv = b * p.Hkv + hk;
    mbar_arrive_expect_tx_w(smem_u32(&bar_q), 2 * Gm::Q_BYTES);
    for (int c = 0; c < NCH; ++c) {
      tma_load_3d_w(sQ + c * BQ * 128, &tmQ, smem_u32(&bar_q), c * 64, q0, bh);
      tma_load_3d_w(sdO + c * BQ * 128, &tmdO, smem_u32(&bar_q), c * 64, q0, bh);
    }
    auto kw = kept_walk<MASKED>(keep, n_kv);
    int jt = kw.first(0);  // key tile of the j-th computed tile
    int nki = 0, nvi = 0;  // K and V tiles issued
    // After an abort (a wait ran out) no further copy is issued, so the
    // drains below cover every copy still in flight.
    for (int j = 0; j < nk; ++j, jt = kw.next(jt)) {
      const int ks = j % KST, vs = j % VST;
      if (j >= KST) mbar_wait(smem_u32(&bar_kempty[ks]), (j / KST - 1) & 1, g, wait_code<11>());
      __syncwarp();
      if (abort_flag) break;
      ++nki;
      mbar_arrive_expect_tx_w(smem_u32(&bar_kfull[ks]), Gm::KV_BYTES);
      for (int c = 0; c < NCH; ++c)
        tma_load_3d_w(sK0 + ks * Gm::KV_BYTES + c * BK * 128, &tmK, smem_u32(&bar_kfull[ks]), c * 64,
                      (j0 + jt) * BK, zkv);
      if (j >= VST) mbar_wait(smem_u32(&bar_vempty[vs]), (j / VST - 1) & 1, g, wait_code<18>());
      __syncwarp();
      if (abort_flag) break;
      ++nvi;
      mbar_arrive_expect_tx_w(smem_u32(&bar_vfull[vs]), Gm::KV_BYTES);
      for (int c = 0; c < NCH; ++c)
        tma_load_3d_w(sV0 + vs * Gm::KV_BYTES + c * BK * 128, &tmV, smem_u32(&bar_vfull[vs]), c * 64,
                      (j0 + jt) * BK, zkv);
    }
    // Q / dO and the last K and V copies issued (a slot is refilled only
    // after its release, so each slot has at most one copy in flight)
    mbar_wait_drain(smem_u32(&bar_q), 0);
    for (int j = (nki > KST ? nki - KST : 0); j < nki; ++j)
      mbar_wait_drain(smem_u32(&bar_kfull[j % KST]), (j / KST) & 1);
    for (int j = (nvi > VST ? nvi - VST : 0); j < nvi; ++j)
      mbar_wait_drain(smem_u32(&bar_vfull[j % VST]), (j / VST) & 1);
    __syncwarp();
  } else if (warp == Gm::MMA_WARP) {
    // ---------------- S / dP issuer (whole warp, one elected lane issues) ----------------
    constexpr uint32_t IDESC_S = make_idesc_f16(128, BK, BF16, false, false);
    const uint64_t dQd = make_sdesc_sw128(sQ, 16, 1024);   // Q, K-major
    const uint64_t dOd = make_sdesc_sw128(sdO, 16, 1024);  // dO, K-major
    const uint64_t dKk = make_sdesc_sw128(sK0, 16, 1024);  // K stage 0, K-major
    const uint64_t dVk = make_sdesc_sw128(sV0, 16, 1024);  // V stage 0, K-major
    mbar_wait(smem_u32(&bar_q), 0, g, wait_code<12>());
    __syncwarp();
    for (int j = 0; j < nk; ++j) {
      const int ks = j % KST, vs = j % VST, buf = j & 1;
      // the dQ MMA of key tile j-2 has read this buffer's dS
      if (j >= 2) mbar_wait(smem_u32(&bar_pfree[buf]), ((j - 2) >> 1) & 1, g, wait_code<19>());
      mbar_wait(smem_u32(&bar_kfull[ks]), (j / KST) & 1, g, wait_code<13>());
      __syncwarp();
      tc_fence_after_sync();
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t qo = (kk >> 2) * (BQ * 128) + (kk & 3) * 32;
        const uint32_t ko = ks * Gm::KV_BYTES + (kk >> 2) * (BK * 128) + (kk & 3) * 32;
        mma_ss_w(tmem + Gm::S_COL + buf * BK, sdesc_add(dQd, qo), sdesc_add(dKk, ko), IDESC_S, kk > 0 ? 1u : 0u);
      }
      mma_commit_w(smem_u32(&bar_kempty[ks]));
      mbar_wait(smem_u32(&bar_vfull[vs]), (j / VST) & 1, g, wait_code<14>());
      __syncwarp();
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t qo = (kk >> 2) * (BQ * 128) + (kk & 3) * 32;
        const uint32_t vo = vs * Gm::KV_BYTES + (kk >> 2) * (BK * 128) + (kk & 3) * 32;
        mma_ss_w(tmem + Gm::DP_COL + buf * BK, sdesc_add(dOd, qo), sdesc_add(dVk, vo), IDESC_S, kk > 0 ? 1u : 0u);
      }
      mma_commit_w(smem_u32(&bar_vempty[vs]));
      mma_commit_w(smem_u32(&bar_sfull[buf]));
    }
    // every MMA this warp issued is complete before tensor memory is released
    mma_commit_w(smem_u32(&bar_sdone));
    mbar_wait_drain(smem_u32(&bar_sdone), 0);
    __syncwarp();
  } else if (warp == Gm::ACC_MMA_WARP) {
    // ---------------- dQ += dS K issuer ----------------
    constexpr uint32_t IDESC_DQ = make_idesc_f16(128, D, BF16, false, true);
    const uint64_t dKm = make_sdesc_sw128(sK0, BK * 128, 1024);  // K stage 0, MN-major
    for (int j = 0; j < nk; ++j) {
      const int ks = j % KST, buf = j & 1;
      mbar_wait(smem_u32(&bar_kfull[ks]), (j / KST) & 1, g, wait_code<10>());
      mbar_wait(smem_u32(&bar_dsready[buf]), (j >> 1) & 1, g, wait_code<15>());
      __syncwarp();
      tc_fence_after_sync();
      // A operand: 16 keys per K step; keys 32h..32h+31 of warpgroup h sit as
      // pairs in columns 32h..32h+15 of the S buffer.
#pragma unroll
      for (int kk = 0; kk < BK / 16; ++kk) {
        const uint32_t acol = Gm::S_COL + buf * BK + (kk >> 1) * 32 + (kk & 1) * 8;
        mma_ts_w(tmem + Gm::DQ_COL, tmem + acol, sdesc_add(dKm, ks * Gm::KV_BYTES + kk * 2048), IDESC_DQ,
                 (j > 0 || kk > 0) ? 1u : 0u);
      }
      mma_commit_w(smem_u32(&bar_pfree[buf]));
      mma_commit_w(smem_u32(&bar_kempty[ks]));
    }
    // every MMA this warp issued is complete (the row threads also wait for
    // it before reading dQ)
    mma_commit_w(smem_u32(&bar_dqdone));
    mbar_wait_drain(smem_u32(&bar_dqdone), 0);
    __syncwarp();
  } else {
    const int quad = warp & 3;   // TMEM lane quadrant (query rows)
    const int half = warp >> 2;  // key columns 32*half .. +31 of each tile
    const int r = quad * 32 + lane;
    const int qi = q0 + r;
    const uint32_t lrow = static_cast<uint32_t>(quad * 32) << 16;
    const float sl2 = p.scale_log2;
    const size_t row = static_cast<size_t>(bh) * p.Lq + qi;
    const float lse_r = qi < p.Lq && dbg_in_range(row, 1, n_qrows, p.status, 10) ? p.lse[row] : 0.f;
    const float dlt_r = qi < p.Lq && dbg_in_range(row, 1, n_qrows, p.status, 11) ? p.delta[row] : 0.f;
    const int lim = CAUSAL ? min((DECODE ? qi % p.qmod : qi) + p.off, p.Lk - 1) : p.Lk - 1;
    const uint64_t sl2x2 = f2_pack(sl2, sl2), nlse2 = f2_pack(-lse_r, -lse_r), dlt2 = f2_pack(dlt_r, dlt_r);
    auto kw = kept_walk<MASKED>(keep, n_kv);
    int jt = kw.first(0);  // key tile of the j-th computed tile
    for (int j = 0; j < nk; ++j, jt = kw.next(jt)) {
      const int buf = j & 1;
      mbar_wait(smem_u32(&bar_sfull[buf]), (j >> 1) & 1, g, wait_code<16>());
      __syncwarp();
      tc_fence_after_sync();
      const int k0 = (j0 + jt) * BK;
      const int kc0 = k0 + half * 32;  // first key of this thread's columns
      const bool need_mask = (CAUSAL && (k0 + BK - 1 > q0 + p.off)) || (k0 + BK > p.Lk);
      const uint32_t scol = tmem + lrow + Gm::S_COL + buf * BK + half * 32;
      uint32_t sr[32], dr[32];
      tmem_ld32(scol, sr);
      tmem_ld32(tmem + lrow + Gm::DP_COL + buf * BK + half * 32, dr);
      tmem_ld_wait(sr);
      reg_fence(dr);
      uint32_t pk[16];
      // two elements per packed instruction
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        float x0, x1;
        f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[2 * i]), __uint_as_float(sr[2 * i + 1])), sl2x2, nlse2), x0, x1);
        float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
        if (need_mask) {
          if (kc0 + 2 * i > lim) p0 = 0.f;
          if (kc0 + 2 * i + 1 > lim) p1 = 0.f;
        }
        const uint64_t d2 = f2_sub(f2_pack(__uint_as_float(dr[2 * i]), __uint_as_float(dr[2 * i + 1])), dlt2);
        float ds0, ds1;
        f2_unpack(f2_mul(f2_pack(p0, p1), d2), ds0, ds1);
        pk[i] = E::pack(ds0, ds1);
      }
      tmem_st16(scol, pk);
      tmem_st_wait();
      tc_fence_before_sync();
      mbar_arrive(smem_u32(&bar_dsready[buf]));
    }
    mbar_wait(smem_u32(&bar_dqdone), 0, g, wait_code<17>());
    __syncwarp();
    tc_fence_after_sync();
    if constexpr (DECODE) {
      // this split's share of row bh * Lq + qi, unscaled
      const size_t x = (static_cast<size_t>(blockIdx.y) * gridDim.x + bh) * p.Lq + qi;
      const size_t n_ws_rows = static_cast<size_t>(gridDim.y) * gridDim.x * p.Lq;  // splits x packed rows
      float* dst = p.ws + x * D;
#pragma unroll 1
      for (int c = half; c < D / 32; c += 2) {
        uint32_t rr[32];
        tmem_ld32(tmem + lrow + Gm::DQ_COL + c * 32, rr);
        tmem_ld_wait(rr);
        if (qi < p.Lq && dbg_in_range(x * D + c * 32, 32, n_ws_rows * D, p.status, 12))
          store_row32_f32(dst + c * 32, rr, 1.f);
      }
    } else {
      typename E::T* dqrow = reinterpret_cast<typename E::T*>(p.dq) + row * D;
#pragma unroll 1
      for (int c = half; c < D / 32; c += 2) {
        uint32_t rr[32];
        if (!MASKED || nk > 0) {  // the same for the whole CTA: tcgen05.ld is warp-collective
          tmem_ld32(tmem + lrow + Gm::DQ_COL + c * 32, rr);
          tmem_ld_wait(rr);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) rr[i] = 0u;  // no kept key tile: dQ = 0
        }
        if (qi < p.Lq && dbg_in_range(row * D + c * 32, 32, n_qrows * D, p.status, 13))
          store_row32<BF16>(dqrow + c * 32, rr, p.scale);
      }
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == Gm::MMA_WARP) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, Gm::TMEM_COLS);
  }
  // Launched behind the dK/dV kernel, this grid may not finish before it:
  // one CTA waiting for it suffices, and holds only its own SM.
  if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) grid_dependency_wait();
}

}  // namespace gbattn
