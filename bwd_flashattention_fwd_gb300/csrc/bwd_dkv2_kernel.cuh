// Backward, dK/dV kernel for head dims up to 128: same mathematics and work
// split as bwd_dkv_kernel.cuh ("feat(attention): complete Flash Attention VJP
// implementation", section "Two-Kernel Design": a CTA owns BK = 128 key rows
// of one (batch, KV head), loops over the G query heads of its group and then
// over the visible query tiles, so dK and dV need no atomics):
//   S^T = K Q^T, dP^T = V dO^T                       (tcgen05, fp32 in TMEM)
//   P^T = exp2(S^T * scale_log2 - lse), dS^T = P^T * (dP^T - delta)
//   dV += P^T dO, dK += dS^T Q                        (tcgen05, A from TMEM)
// and finally dK is scaled by `scale`.
//
// Layout for throughput.  An MMA with both operands in shared memory at N = 64
// needs more shared-memory bandwidth than the SM has, and K does not change
// over the CTA's loop, so the row threads copy K once into tensor memory and
// S^T = K Q^T reads only Q from shared memory.  Tensor memory (512 columns):
// dK, dV (128 each), K (D/2 columns of 16-bit pairs), one S^T buffer and two
// dP^T buffers of 64 columns.  The row threads write P^T and dS^T (16-bit
// pairs) over the dP^T columns they have read.  Two warps issue the MMAs,
// each in an order that needs no completion round trip (tcgen05 MMAs of one
// issuing thread execute in issue order):
//   * the S warp issues S^T(i+1) as soon as every row thread has loaded S^T(i)
//     into registers ("S free" barrier), so it runs while the rows compute;
//   * the accumulate warp issues dV(i) and dK(i), then dP^T(i+2) into the same
//     dP^T buffer, behind the MMAs that read P^T(i) and dS^T(i) from it.
//
// Warp roles (352 threads): warps 0-7 row threads -- warp w owns TMEM lanes
// 32*(w%4)..+31 (key rows) and query columns 32*(w/4)..+31 of each tile, and
// copies D/2 columns of its key rows into tensor memory; warp 8 producer (TMA
// for the V tile and the Q/dO tiles, plain loads for the per-query lse/delta
// values); warp 9 issues S^T and owns the TMEM allocation; warp 10 issues
// dV, dK and dP^T.  A share of the exponentials of the row warps on the
// sub-partitions of warps 9 and 10 can be evaluated with a polynomial on the
// FMA pipe (ex2_poly2; GBATTN_DKV_POLY_Q1 / _Q2); none measured fastest.
// (With equal shares, this three-way dispatch measured ~3% faster than a
// single call.)
//
// MASKED: block-sparse variant ("feat(attention): complete Flash Attention
// VJP implementation", section "Sparse Block Masks": the dK/dV kernel skips
// the query blocks whose mask entry is zero).  The CTA's 128 keys are one
// mask block and a query tile half of a 128-row block; skipped query tiles
// are neither loaded nor computed, and every warp walks the same list of kept
// tiles.  A key tile with no kept query tile writes dK = dV = 0.
//
#pragma once

#include <type_traits>

#include "kernel_common.cuh"

namespace gbattn {

template <int D>
struct Dkv2Geom {
  static constexpr int BK = 128;  // key rows per CTA (MMA M)
  static constexpr int BQ = 64;   // query rows per iteration (MMA N of S^T)
  static constexpr int NCH = n_chunks(D);
  static constexpr int V_BYTES = NCH * BK * 128;
  static constexpr int Q_BYTES = NCH * BQ * 128;
  static constexpr int STAGES_FIT = (kMaxDynSmem - kSmemReserve - 1024 - V_BYTES) / (2 * Q_BYTES);
  static constexpr int STAGES = STAGES_FIT > 5 ? 5 : STAGES_FIT;
  static constexpr int SMEM_BYTES = 1024 + V_BYTES + STAGES * 2 * Q_BYTES;
  static constexpr int DK_COL = 0, DV_COL = 128, K_COL = 256, ST_COL = 320, DPT_COL = 384;  // dP^T: 2 x 64
  static constexpr int TMEM_COLS = 512;
  static constexpr int NUM_COMPUTE_WARPS = 8;
  static constexpr int NCT = 32 * NUM_COMPUTE_WARPS;
  static constexpr int PRODUCER_WARP = NUM_COMPUTE_WARPS;
  static constexpr int S_MMA_WARP = NUM_COMPUTE_WARPS + 1;
  static constexpr int ACC_MMA_WARP = NUM_COMPUTE_WARPS + 2;
  static constexpr int NUM_THREADS = 32 * (NUM_COMPUTE_WARPS + 3);
  // element pairs (of 16 per thread and query tile) whose exponentials use the
  // polynomial, on the sub-partition of the S warp (1) and of the accumulate
  // warp (2)
#ifndef GBATTN_DKV_POLY_Q1
  static constexpr int POLY_Q1 = 0;
#else
  static constexpr int POLY_Q1 = GBATTN_DKV_POLY_Q1;
#endif
#ifndef GBATTN_DKV_POLY_Q2
  static constexpr int POLY_Q2 = 0;
#else
  static constexpr int POLY_Q2 = GBATTN_DKV_POLY_Q2;
#endif
  static_assert(D <= 128, "dK, dV, K and the S^T / dP^T buffers fill TMEM at D = 128");
  // the S warp works on tile i+1 and the accumulate warp loads dP^T(i+2) while
  // tile i is in use
  static_assert(STAGES >= 3, "shared memory budget");
  static_assert(POLY_Q1 >= 0 && POLY_Q1 <= 16 && POLY_Q2 >= 0 && POLY_Q2 <= 16, "polynomial share");
};

template <int D, bool BF16, bool CAUSAL, bool MASKED>
__global__ void __launch_bounds__(Dkv2Geom<D>::NUM_THREADS, 1)
    attn_bwd_dkv2_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmV,
                         const __grid_constant__ CUtensorMap tmdO, const void* __restrict__ k, const BwdParams p) {
  using Gm = Dkv2Geom<D>;
  using E = Elem<BF16>;
  constexpr int BQ = Gm::BQ, BK = Gm::BK, NCH = Gm::NCH, ST = Gm::STAGES, NCT = Gm::NCT;

  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t bar_v, bar_kready, bar_stfull[ST], bar_stempty[ST], bar_sfull, bar_sfree, bar_dpfull[2],
      bar_pready[2], bar_accdone, bar_sdone;
  __shared__ __align__(16) float nlse_s[ST][BQ];  // -lse per query column
  __shared__ __align__(16) float dlt_s[ST][BQ];
  __shared__ uint32_t tmem_slot;
  __shared__ volatile int abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t sV = sbase;
  const uint32_t sQ0 = sbase + Gm::V_BYTES;
  const uint32_t sdO0 = sQ0 + ST * Gm::Q_BYTES;

  const int bhk = blockIdx.x;  // b * Hkv + hk
  const int b = bhk / p.Hkv, hk = bhk - b * p.Hkv;
  const int kt = blockIdx.y;
  const int k0 = kt * BK;
  const int qt_start = CAUSAL ? max(0, k0 - p.off) / BQ : 0;
  static_assert(BK == kMaskBlock && 2 * BQ == kMaskBlock, "key tile = mask block, query tile = half a block");
  // query tile qt is computed (block mask)
  auto keep = [&](int qt) { return !MASKED || mask_keep(p, qt >> 1, kt); };
  const WaitGuard g{&abort_flag, p.status, p.limit_ns};
  // extents for the debug build's index checks: rows of q / dq / lse /
  // delta, of dk / dv, and of the k / v buffers (pitch kv_pitch per head)
  [[maybe_unused]] const size_t n_qrows = static_cast<size_t>(p.B) * p.Hq * p.Lq;
  [[maybe_unused]] const size_t n_krows = static_cast<size_t>(p.B) * p.Hkv * p.Lk;
  [[maybe_unused]] const size_t n_kvbuf = (static_cast<size_t>(p.B) * p.Hkv - 1) * p.kv_pitch + p.Lk;

  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(smem_u32(&bar_v), 1);
    mbar_init(smem_u32(&bar_kready), NCT);
    for (int s = 0; s < ST; ++s) {
      mbar_init(smem_u32(&bar_stfull[s]), 33);  // TMA expect_tx arrive + 32 producer lanes
      mbar_init(smem_u32(&bar_stempty[s]), 2);  // S^T (S warp) and dP^T, dV, dK (accumulate warp)
    }
    mbar_init(smem_u32(&bar_sfull), 1);
    mbar_init(smem_u32(&bar_sfree), NCT);
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&bar_dpfull[i]), 1);
      mbar_init(smem_u32(&bar_pready[i]), NCT);
    }
    mbar_init(smem_u32(&bar_accdone), 1);
    mbar_init(smem_u32(&bar_sdone), 1);
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
  // Launched behind the delta kernel as a programmatic dependent, this grid
  // may start while that kernel finishes: it reads nothing in global memory
  // (lse, delta, the inputs, the block mask) before every earlier kernel on
  // the stream has completed.  Only then may a dQ kernel launched behind this
  // one start filling the SMs this grid frees (it reads lse and delta, but
  // none of this grid's outputs, without waiting itself).
  grid_dependency_wait();
  if (threadIdx.x == 0) grid_launch_dependents();
  // (query head, computed query tile) iterations; every warp counts them itself
  const int n_iter = p.G * count_kept<MASKED>(keep, qt_start, p.n_qtiles);

  if (warp == Gm::PRODUCER_WARP) {
    // ---------------- producer (whole warp) ----------------
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmdO);
      tma_prefetch_desc(&tmV);
    }
    __syncwarp();
    mbar_arrive_expect_tx_w(smem_u32(&bar_v), Gm::V_BYTES);
    for (int c = 0; c < NCH; ++c) tma_load_3d_w(sV + c * BK * 128, &tmV, smem_u32(&bar_v), c * 64, k0, bhk);
    RingPos<ST> st;                  // stage of iteration it
    auto qw = kept_walk<MASKED>(keep, p.n_qtiles);
    int gi = 0, qtile = qw.first(qt_start);  // query head in the group and query tile of iteration it
    int ni = 0;  // stages issued; after an abort (a wait ran out) no further copy is issued
    for (int it = 0; it < n_iter; ++it, st.next()) {
      const int s = st.slot;
      if (it >= ST) mbar_wait(smem_u32(&bar_stempty[s]), st.phase ^ 1u, g, wait_code<81>());
      __syncwarp();
      if (abort_flag) break;
      ++ni;
      const int q0 = qtile * BQ;
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
        nlse_s[s][c] = qi < p.Lq && dbg_in_range(row, 1, n_qrows, p.status, 14) ? -p.lse[row] : -INFINITY;
        dlt_s[s][c] = qi < p.Lq && dbg_in_range(row, 1, n_qrows, p.status, 15) ? p.delta[row] : 0.f;
      }
      mbar_arrive(smem_u32(&bar_stfull[s]));
      qtile = qw.next(qtile);
      if (qtile >= p.n_qtiles) qtile = qw.first(qt_start), ++gi;
    }
    // V and the last ST stages issued (a stage is refilled only after its
    // release, so each holds at most one copy in flight)
    mbar_wait_drain(smem_u32(&bar_v), 0);
    for (int it = (ni > ST ? ni - ST : 0); it < ni; ++it)
      mbar_wait_drain(smem_u32(&bar_stfull[it % ST]), (it / ST) & 1);
  } else if (warp == Gm::S_MMA_WARP) {
    // ---------------- S^T = K Q^T issuer (A operand K from tensor memory) ----------------
    constexpr uint32_t IDESC_S = make_idesc_f16(128, BQ, BF16, false, false);
    const uint64_t dQk = make_sdesc_sw128(sQ0, 16, 1024);  // Q stage 0, K-major
    mbar_wait(smem_u32(&bar_kready), 0, g, wait_code<82>());
    __syncwarp();
    tc_fence_after_sync();
    RingPos<ST> st;  // stage of iteration it
    for (int it = 0; it < n_iter; ++it, st.next()) {
      const int s = st.slot;
      // every row thread has loaded S^T(it-1) from the buffer
      if (it >= 1) mbar_wait(smem_u32(&bar_sfree), (it - 1) & 1, g, wait_code<83>());
      mbar_wait(smem_u32(&bar_stfull[s]), st.phase, g, wait_code<84>());
      __syncwarp();
      tc_fence_after_sync();
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t qo = s * Gm::Q_BYTES + (kk >> 2) * (BQ * 128) + (kk & 3) * 32;
        mma_ts_w(tmem + Gm::ST_COL, tmem + Gm::K_COL + kk * 8, sdesc_add(dQk, qo), IDESC_S, kk > 0 ? 1u : 0u);
      }
      mma_commit_w(smem_u32(&bar_sfull));
      mma_commit_w(smem_u32(&bar_stempty[s]));
    }
    // every MMA this warp issued is complete before tensor memory is released
    mma_commit_w(smem_u32(&bar_sdone));
    mbar_wait_drain(smem_u32(&bar_sdone), 0);
    __syncwarp();
  } else if (warp == Gm::ACC_MMA_WARP) {
    // ---------------- dV += P^T dO, dK += dS^T Q and dP^T = V dO^T issuer ----------------
    constexpr uint32_t IDESC_S = make_idesc_f16(128, BQ, BF16, false, false);
    constexpr uint32_t IDESC_ACC = make_idesc_f16(128, D, BF16, false, true);
    const uint64_t dV = make_sdesc_sw128(sV, 16, 1024);             // V tile, K-major
    const uint64_t dOk = make_sdesc_sw128(sdO0, 16, 1024);          // dO stage 0, K-major
    const uint64_t dQm = make_sdesc_sw128(sQ0, BQ * 128, 1024);     // Q stage 0, MN-major
    const uint64_t dOm = make_sdesc_sw128(sdO0, BQ * 128, 1024);    // dO stage 0, MN-major
    mbar_wait(smem_u32(&bar_v), 0, g, wait_code<85>());
    __syncwarp();
    RingPos<ST> st, st_dp;  // stages of the next dV / dK and of the next dP^T iteration
    auto issue_dp = [&](int it) {
      const int s = st_dp.slot, buf = it & 1;
      mbar_wait(smem_u32(&bar_stfull[s]), st_dp.phase, g, wait_code<86>());
      __syncwarp();
      tc_fence_after_sync();
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t vo = (kk >> 2) * (BK * 128) + (kk & 3) * 32;
        const uint32_t qo = s * Gm::Q_BYTES + (kk >> 2) * (BQ * 128) + (kk & 3) * 32;
        mma_ss_w(tmem + Gm::DPT_COL + buf * BQ, sdesc_add(dV, vo), sdesc_add(dOk, qo), IDESC_S, kk > 0 ? 1u : 0u);
      }
      mma_commit_w(smem_u32(&bar_dpfull[buf]));
      st_dp.next();
    };
    for (int it = 0; it < 2 && it < n_iter; ++it) issue_dp(it);
    for (int it = 0; it < n_iter; ++it, st.next()) {
      const int s = st.slot, buf = it & 1;
      mbar_wait(smem_u32(&bar_pready[buf]), (it >> 1) & 1, g, wait_code<87>());
      __syncwarp();
      tc_fence_after_sync();
      // A operands: 16 queries per K step; the warps of query half h hold P^T
      // of queries 32h..32h+31 as pairs in columns 32h..32h+15 of the buffer
      // and dS^T in columns 32h+16..32h+31.
#pragma unroll
      for (int kk = 0; kk < BQ / 16; ++kk) {
        const uint32_t acol = Gm::DPT_COL + buf * BQ + (kk >> 1) * 32 + (kk & 1) * 8;
        const uint32_t bo = s * Gm::Q_BYTES + kk * 2048;
        mma_ts_w(tmem + Gm::DV_COL, tmem + acol, sdesc_add(dOm, bo), IDESC_ACC, (it > 0 || kk > 0) ? 1u : 0u);
        mma_ts_w(tmem + Gm::DK_COL, tmem + acol + 16, sdesc_add(dQm, bo), IDESC_ACC, (it > 0 || kk > 0) ? 1u : 0u);
      }
      // this warp's dP^T(it), dV(it) and dK(it) are its last reads of the stage
      mma_commit_w(smem_u32(&bar_stempty[s]));
      // dP^T(it+2) overwrites the buffer behind the MMAs that read P^T / dS^T
      if (it + 2 < n_iter) issue_dp(it + 2);
    }
    // every MMA this warp issued is complete before tensor memory is
    // released (the row threads also wait for it before reading dK, dV)
    mma_commit_w(smem_u32(&bar_accdone));
    mbar_wait_drain(smem_u32(&bar_accdone), 0);
    __syncwarp();
  } else {
    // ---------------- key-row threads ----------------
    const int quad = warp & 3;   // TMEM lane quadrant (key rows)
    const int half = warp >> 2;  // query columns 32*half .. +31
    const int r = quad * 32 + lane;
    const int kj = k0 + r;
    const uint32_t lrow = static_cast<uint32_t>(quad * 32) << 16;
    const float sl2 = p.scale_log2;
    const uint64_t sl2x2 = f2_pack(sl2, sl2);
    const int qmin = kj - p.off;  // causal: queries below this index cannot see key kj
    const size_t krow = static_cast<size_t>(bhk) * p.Lk + kj;  // row of dK / dV
    const size_t kin = static_cast<size_t>(bhk) * p.kv_pitch + kj;  // row of K
    // K row into tensor memory: this warp copies columns [half*D/2,
    // (half+1)*D/2) of its 32 key rows (zeros past Lk), as 16-bit pairs.
    {
      constexpr int HALF = D / 2;   // elements per thread
      constexpr int NV = HALF / 8;  // 16-byte loads per thread
      const uint4* src =
          reinterpret_cast<const uint4*>(reinterpret_cast<const typename E::T*>(k) + kin * D + half * HALF);
      uint32_t ka[HALF / 2];
#pragma unroll
      for (int v = 0; v < NV; ++v) {
        uint4 x = make_uint4(0u, 0u, 0u, 0u);
        if (kj < p.Lk && dbg_in_range(kin * D + half * HALF + 8 * v, 8, n_kvbuf * D, p.status, 16)) x = src[v];
        ka[4 * v + 0] = x.x, ka[4 * v + 1] = x.y, ka[4 * v + 2] = x.z, ka[4 * v + 3] = x.w;
      }
      // HALF / 2 packed columns: 16, 24 or 32 (D = 64, 96, 128)
#pragma unroll
      for (int c = 0; c + 16 <= HALF / 2; c += 16) {
        uint32_t t16[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) t16[i] = ka[c + i];
        tmem_st16(tmem + lrow + Gm::K_COL + half * (HALF / 2) + c, t16);
      }
      if constexpr ((HALF / 2) % 16 == 8) {
        constexpr int c = HALF / 2 - 8;
        uint32_t t8[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) t8[i] = ka[c + i];
        tmem_st8(tmem + lrow + Gm::K_COL + half * (HALF / 2) + c, t8);
      }
      tmem_st_wait();
      tc_fence_before_sync();
      mbar_arrive(smem_u32(&bar_kready));
    }
    RingPos<ST> st;             // stage of iteration it
    auto qw = kept_walk<MASKED>(keep, p.n_qtiles);
    int qtile = qw.first(qt_start);  // query tile of iteration it
    for (int it = 0; it < n_iter; ++it, st.next()) {
      const int s = st.slot, buf = it & 1;
      const int q0 = qtile * BQ;
      qtile = qw.next(qtile);
      if (qtile >= p.n_qtiles) qtile = qw.first(qt_start);
      mbar_wait(smem_u32(&bar_stfull[s]), st.phase, g, wait_code<88>());
      mbar_wait(smem_u32(&bar_sfull), it & 1, g, wait_code<89>());
      mbar_wait(smem_u32(&bar_dpfull[buf]), (it >> 1) & 1, g, wait_code<90>());
      __syncwarp();
      tc_fence_after_sync();
      const bool need_mask = CAUSAL && (q0 < k0 + BK - 1 - p.off);
      const uint32_t dcol = tmem + lrow + Gm::DPT_COL + buf * BQ + half * 32;
      uint32_t sr[32], dr[32];
      tmem_ld32(tmem + lrow + Gm::ST_COL + half * 32, sr);
      tmem_ld32(dcol, dr);
      tmem_ld_wait(sr);
      reg_fence(dr);
      // S^T(it) is in registers: the S warp may overwrite the buffer
      tc_fence_before_sync();
      mbar_arrive(smem_u32(&bar_sfree));
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
          f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[c0]), __uint_as_float(sr[c0 + 1])), sl2x2, nlse_row[i]), x0,
                    x1);
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
          const uint64_t d2 = f2_sub(f2_pack(__uint_as_float(dr[c0]), __uint_as_float(dr[c0 + 1])), dlt_row[i]);
          float ds0, ds1;
          f2_unpack(f2_mul(f2_pack(p0, p1), d2), ds0, ds1);
          dk[i] = E::pack(ds0, ds1);
        }
      };
      if (quad == 1)  // sub-partition of the S warp (9)
        pds_tile(std::integral_constant<int, Gm::POLY_Q1>{});
      else if (quad == 2)  // sub-partition of the accumulate warp (10)
        pds_tile(std::integral_constant<int, Gm::POLY_Q2>{});
      else
        pds_tile(std::integral_constant<int, 0>{});
      tmem_st16(dcol, pk);
      tmem_st16(dcol + 16, dk);
      tmem_st_wait();
      tc_fence_before_sync();
      mbar_arrive(smem_u32(&bar_pready[buf]));
    }
    mbar_wait(smem_u32(&bar_accdone), 0, g, wait_code<91>());
    __syncwarp();
    tc_fence_after_sync();
    // epilogue: warpgroup `half` writes output columns [half*D/2, (half+1)*D/2)
    typename E::T* dkrow = reinterpret_cast<typename E::T*>(p.dk) + krow * D;
    typename E::T* dvrow = reinterpret_cast<typename E::T*>(p.dv) + krow * D;
#pragma unroll 1
    for (int c = half; c < D / 32; c += 2) {
      uint32_t rr[32];
      if (n_iter > 0) {
        tmem_ld32(tmem + lrow + Gm::DK_COL + c * 32, rr);
        tmem_ld_wait(rr);
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) rr[i] = 0u;  // no kept query tile: dK = dV = 0
      }
      if (kj < p.Lk && dbg_in_range(krow * D + c * 32, 32, n_krows * D, p.status, 17))
        store_row32<BF16>(dkrow + c * 32, rr, p.scale);
      if (n_iter > 0) {
        tmem_ld32(tmem + lrow + Gm::DV_COL + c * 32, rr);
        tmem_ld_wait(rr);
      }
      if (kj < p.Lk && dbg_in_range(krow * D + c * 32, 32, n_krows * D, p.status, 18))
        store_row32<BF16>(dvrow + c * 32, rr, 1.f);
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
