// Forward attention with saved base-2 log-sum-exp.
//
// One CTA owns a tile of BQ = 128 query rows of one (batch, query head) and
// walks the visible key tiles with an online softmax ("When the Bottleneck
// Moved", section 3: m_new = max(m_old, rowmax S), alpha = exp(m_old - m_new),
// l_new = alpha l_old + rowsum p, acc_new = alpha acc_old + p V, then
// O = acc / l and L = m + log l), kept in the log2 domain ("feat(attention):
// complete Flash Attention VJP implementation", section "Background":
// P = exp2(S * scale_log2 - LSE)).
//
// Warp roles (224 threads):
//   warps 0-3  softmax: thread t of warp w owns query row 32w+t, which is TMEM
//              lane 32w+t of every accumulator;
//   warp 4     TMA producer: Q once, then K and V tiles into their rings;
//   warp 5     issues S = Q K^T (one thread) and owns the TMEM allocation;
//   warp 6     issues O += P V.
// Two issuing warps halve the serial barrier waits and commits per key tile
// of each; S of tile j+2 is issued as soon as the softmax warps have loaded
// S of tile j, so the score products run two tiles ahead of P V.
// Tensor memory (512 columns): O (D columns, fp32), two S buffers (BK columns
// each, fp32) and two P buffers (BK/2 columns, bf16/fp16 pairs).  S_j = Q K_j^T
// runs on the tensor cores while the softmax warps turn S_{j-1} into P_{j-1};
// O += P_j V_j reads P straight from tensor memory.  A row keeps its
// reference maximum until a tile raises the row maximum by more than 8 (log2
// units), so the 256-column O accumulator is rescaled only on those rare
// tiles; O / l and lse = m + log2 l use the same reference, so the result is
// exact in exact arithmetic.
//
// DECODE (short query lengths): the G query heads x Lq rows of one KV head
// (consecutive in the [B, Hq, Lq, D] layout) form one packed tile; packed row
// r is query r % Lq.  CTA (x, y) covers key tiles [y*split_tiles, ...) of
// KV head x and writes each row's partial O (normalised by its own sum) and
// partial base-2 log-sum-exp in fp32; a combine kernel merges the splits
// (the online-softmax merge of "When the Bottleneck Moved", section 3, applied
// across CTAs).  A row may see no key of its split: its partial lse is -inf.
//
// MASKED: block-sparse variant ("feat(attention): complete Flash Attention
// VJP implementation", section "Sparse Block Masks"): the query tile is one
// 128-row mask block; key tiles whose mask block is zero are neither loaded
// nor computed (found 32 at a time by a warp ballot), and a row that sees no
// key gets O = 0 and lse = +inf.
#pragma once

#include "kernel_common.cuh"

namespace gbattn {

template <int D>
struct FwdGeom {
  static constexpr int BQ = 128;
  static constexpr int BK = (D == 256) ? 64 : 128;
  static constexpr int NCH = n_chunks(D);
  static constexpr int Q_BYTES = NCH * BQ * 128;
  static constexpr int KV_BYTES = NCH * BK * 128;
  // K and V tiles have rings of their own: a K tile is free once S = Q K^T
  // has read it, a V tile only after P V, so the K ring runs further ahead.
  // (The kernel's static shared memory, barriers only, stays under 1 KB.)
  static constexpr int SLOTS = (kMaxDynSmem - 1024 - 1024 - Q_BYTES) / KV_BYTES;
  static constexpr int KSTAGES = SLOTS - 2 > 4 ? 4 : SLOTS - 2;
  static constexpr int VSTAGES = SLOTS - KSTAGES > 4 ? 4 : SLOTS - KSTAGES;
  static constexpr int SMEM_BYTES = 1024 + Q_BYTES + (KSTAGES + VSTAGES) * KV_BYTES;
  static constexpr int O_COL = 0;
  static constexpr int S_COL0 = (D <= 128) ? 128 : 256;
  static constexpr int S_COL1 = S_COL0 + BK;
  static constexpr int P_COL0 = S_COL1 + BK;
  static constexpr int P_COL1 = P_COL0 + BK / 2;
  static constexpr int TMEM_COLS = 512;
  static constexpr int NUM_THREADS = 224;
  static constexpr float TAU = 8.0f;  // lazy-rescaling threshold (log2 units)
  static_assert(KSTAGES >= 2 && VSTAGES >= 2, "need double-buffered K and V rings");
  static_assert(P_COL1 + BK / 2 <= TMEM_COLS, "tensor memory budget");
  // Tensor memory left over (64 columns at D = 256) holds the first K steps
  // of Q as 16-bit pairs: those S = Q K^T steps read A from tensor memory,
  // the rest from shared memory (an MMA with both operands in shared memory
  // at N = 64 is bound by shared-memory bandwidth).
  static constexpr int QT_COL = P_COL1 + BK / 2;
  static constexpr int QT_STEPS = (TMEM_COLS - QT_COL) / 8 < D / 16 ? (TMEM_COLS - QT_COL) / 8 : D / 16;
};

template <int D, bool BF16, bool CAUSAL, bool DECODE = false, bool MASKED = false>
__global__ void __launch_bounds__(FwdGeom<D>::NUM_THREADS, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const FwdParams p) {
  using Gm = FwdGeom<D>;
  using E = Elem<BF16>;
  constexpr int BQ = Gm::BQ, BK = Gm::BK, NCH = Gm::NCH, KST = Gm::KSTAGES, VST = Gm::VSTAGES;

  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t bar_q, bar_kfull[KST], bar_kempty[KST], bar_vfull[VST], bar_vempty[VST], bar_sfull[2],
      bar_sfree[2], bar_pready[2], bar_pvdone[2], bar_drain[2], bar_qready;
  __shared__ uint32_t tmem_slot;
  __shared__ volatile int abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t sQ = sbase;
  const uint32_t sK0 = sQ + Gm::Q_BYTES;
  const uint32_t sV0 = sK0 + KST * Gm::KV_BYTES;

  const int bh = blockIdx.x;  // b * Hq + hq (decode: b * Hkv + hk, with Hq = Hkv, G = 1)
  const int b = bh / p.Hq, hq = bh - b * p.Hq;
  const int hk = hq / p.G;
  const int qt = DECODE ? 0 : p.n_qtiles - 1 - static_cast<int>(blockIdx.y);  // heaviest tiles first
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
  // extents for the debug build's index checks: rows of q / o / lse
  [[maybe_unused]] const size_t n_qrows = static_cast<size_t>(p.B) * p.Hq * p.Lq;

  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(smem_u32(&bar_q), 1);
    mbar_init(smem_u32(&bar_qready), 128);
    for (int s = 0; s < KST; ++s) {
      mbar_init(smem_u32(&bar_kfull[s]), 1);
      mbar_init(smem_u32(&bar_kempty[s]), 1);
    }
    for (int s = 0; s < VST; ++s) {
      mbar_init(smem_u32(&bar_vfull[s]), 1);
      mbar_init(smem_u32(&bar_vempty[s]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&bar_sfull[i]), 1);
      mbar_init(smem_u32(&bar_sfree[i]), 128);
      mbar_init(smem_u32(&bar_pready[i]), 128);
      mbar_init(smem_u32(&bar_pvdone[i]), 1);
      mbar_init(smem_u32(&bar_drain[i]), 1);
    }
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
    // ---------------- TMA producer (whole warp, one elected lane issues) ----------------
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
    }
    __syncwarp();
    const int zkv = b * p.Hkv + hk;
    mbar_arrive_expect_tx_w(smem_u32(&bar_q), Gm::Q_BYTES);
    for (int c = 0; c < NCH; ++c) tma_load_3d_w(sQ + c * BQ * 128, &tmQ, smem_u32(&bar_q), c * 64, q0, bh);
    RingPos<KST> kp;
    RingPos<VST> vp;
    auto kw = kept_walk<MASKED>(keep, n_kv);
    int jt = kw.first(0);  // key tile of the j-th computed tile
    int nki = 0, nvi = 0;  // K and V tiles issued
    // After an abort (a wait ran out) no further copy is issued, so the
    // drains below cover every copy still in flight.
    for (int j = 0; j < nk; ++j, jt = kw.next(jt), kp.next(), vp.next()) {
      const int ks = kp.slot, vs = vp.slot;
      if (j >= KST) mbar_wait(smem_u32(&bar_kempty[ks]), kp.phase ^ 1u, g, wait_code<1>());
      __syncwarp();
      if (abort_flag) break;
      mbar_arrive_expect_tx_w(smem_u32(&bar_kfull[ks]), Gm::KV_BYTES);
      for (int c = 0; c < NCH; ++c)
        tma_load_3d_w(sK0 + ks * Gm::KV_BYTES + c * BK * 128, &tmK, smem_u32(&bar_kfull[ks]), c * 64, (j0 + jt) * BK,
                      zkv);
      ++nki;
      if (j >= VST) mbar_wait(smem_u32(&bar_vempty[vs]), vp.phase ^ 1u, g, wait_code<9>());
      __syncwarp();
      if (abort_flag) break;
      mbar_arrive_expect_tx_w(smem_u32(&bar_vfull[vs]), Gm::KV_BYTES);
      for (int c = 0; c < NCH; ++c)
        tma_load_3d_w(sV0 + vs * Gm::KV_BYTES + c * BK * 128, &tmV, smem_u32(&bar_vfull[vs]), c * 64, (j0 + jt) * BK,
                      zkv);
      ++nvi;
    }
    // Do not leave the CTA while a copy may still be landing: Q and the last
    // K and V copies issued (a slot is refilled only after its release, so
    // each slot has at most one copy in flight).
    mbar_wait_drain(smem_u32(&bar_q), 0);
    for (int j = (nki > KST ? nki - KST : 0); j < nki; ++j)
      mbar_wait_drain(smem_u32(&bar_kfull[j % KST]), (j / KST) & 1);
    for (int j = (nvi > VST ? nvi - VST : 0); j < nvi; ++j)
      mbar_wait_drain(smem_u32(&bar_vfull[j % VST]), (j / VST) & 1);
    __syncwarp();
  } else if (warp == 5) {
    // ---------------- S = Q K^T issuer (whole warp, one elected lane issues) ----------------
    constexpr uint32_t IDESC_QK = make_idesc_f16(128, BK, BF16, false, false);
    const uint64_t dQd = make_sdesc_sw128(sQ, 16, 1024);   // Q, K-major
    const uint64_t dKk = make_sdesc_sw128(sK0, 16, 1024);  // K stage 0, K-major
    // Q in shared memory, and its first QT_STEPS K steps in tensor memory
    if constexpr (Gm::QT_STEPS > 0)
      mbar_wait(smem_u32(&bar_qready), 0, g, wait_code<93>());
    else
      mbar_wait(smem_u32(&bar_q), 0, g, wait_code<2>());
    for (int j = 0; j < nk; ++j) {  // j: computed tiles so far
      const int s = j % KST;
      // the softmax warps have loaded S of tile j-2 from this buffer
      if (j >= 2) mbar_wait(smem_u32(&bar_sfree[j & 1]), ((j - 2) >> 1) & 1, g, wait_code<4>());
      mbar_wait(smem_u32(&bar_kfull[s]), (j / KST) & 1, g, wait_code<3>());
      __syncwarp();
      tc_fence_after_sync();
      const uint32_t d = tmem + ((j & 1) ? Gm::S_COL1 : Gm::S_COL0);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t qo = (kk >> 2) * (BQ * 128) + (kk & 3) * 32;
        const uint32_t ko = s * Gm::KV_BYTES + (kk >> 2) * (BK * 128) + (kk & 3) * 32;
        if (kk < Gm::QT_STEPS)
          mma_ts_w(d, tmem + Gm::QT_COL + kk * 8, sdesc_add(dKk, ko), IDESC_QK, kk > 0 ? 1u : 0u);
        else
          mma_ss_w(d, sdesc_add(dQd, qo), sdesc_add(dKk, ko), IDESC_QK, kk > 0 ? 1u : 0u);
      }
      mma_commit_w(smem_u32(&bar_sfull[j & 1]));
      mma_commit_w(smem_u32(&bar_kempty[s]));  // S_j was K_j's only reader
    }
    // every MMA this warp issued is complete before tensor memory is released
    mma_commit_w(smem_u32(&bar_drain[0]));
    mbar_wait_drain(smem_u32(&bar_drain[0]), 0);
    __syncwarp();
  } else if (warp == 6) {
    // ---------------- O += P V issuer ----------------
    constexpr uint32_t IDESC_PV = make_idesc_f16(128, D, BF16, false, true);
    const uint64_t dVm = make_sdesc_sw128(sV0, BK * 128, 1024);  // V stage 0, MN-major
    for (int j = 0; j < nk; ++j) {
      const int sp = j % VST;
      mbar_wait(smem_u32(&bar_pready[j & 1]), (j >> 1) & 1, g, wait_code<5>());
      mbar_wait(smem_u32(&bar_vfull[sp]), (j / VST) & 1, g, wait_code<32>());
      __syncwarp();
      tc_fence_after_sync();
      const uint32_t pcol = tmem + ((j & 1) ? Gm::P_COL1 : Gm::P_COL0);
#pragma unroll
      for (int kk = 0; kk < BK / 16; ++kk)
        mma_ts_w(tmem + Gm::O_COL, pcol + kk * 8, sdesc_add(dVm, sp * Gm::KV_BYTES + kk * 2048), IDESC_PV,
                 (j > 0 || kk > 0) ? 1u : 0u);
      mma_commit_w(smem_u32(&bar_vempty[sp]));
      mma_commit_w(smem_u32(&bar_pvdone[j & 1]));  // P buffer j&1 free; O includes tile j
    }
    mma_commit_w(smem_u32(&bar_drain[1]));
    mbar_wait_drain(smem_u32(&bar_drain[1]), 0);
    __syncwarp();
  } else {
    // ---------------- softmax warps ----------------
    const int r = warp * 32 + lane;
    const int qi = q0 + r;
    const uint32_t lrow = static_cast<uint32_t>(warp * 32) << 16;
    const float sl2 = p.scale_log2;
    // last visible key of this row (inclusive)
    const int lim = CAUSAL ? min((DECODE ? qi % p.qmod : qi) + p.off, p.Lk - 1) : p.Lk - 1;
    if constexpr (Gm::QT_STEPS > 0) {
      // this row's first 16 * QT_STEPS elements of Q from shared memory (TMA
      // layout: 64-column chunks of 128-byte rows, 16-byte units swizzled by
      // row % 8) into tensor memory as 16-bit pairs
      constexpr int NQ = 16 * Gm::QT_STEPS;  // elements
      mbar_wait(smem_u32(&bar_q), 0, g, wait_code<92>());
      uint32_t qa[NQ / 2];
#pragma unroll
      for (int v = 0; v < NQ / 8; ++v) {
        const int e = 8 * v;
        const uint4 x = ld_shared_v4(sQ + (e / 64) * (BQ * 128) + r * 128 + ((((e % 64) / 8) ^ (r & 7)) * 16));
        qa[4 * v + 0] = x.x, qa[4 * v + 1] = x.y, qa[4 * v + 2] = x.z, qa[4 * v + 3] = x.w;
      }
#pragma unroll
      for (int c = 0; c < NQ / 2; c += 16) {
        uint32_t t16[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) t16[i] = qa[c + i];
        tmem_st16(tmem + lrow + Gm::QT_COL + c, t16);
      }
      tmem_st_wait();
      tc_fence_before_sync();
      mbar_arrive(smem_u32(&bar_qready));
    }
    float m = -INFINITY, l = 0.f;
    auto kw = kept_walk<MASKED>(keep, n_kv);
    int jt = kw.first(0);  // key tile of the j-th computed tile
    for (int j = 0; j < nk; ++j, jt = kw.next(jt)) {
      mbar_wait(smem_u32(&bar_sfull[j & 1]), (j >> 1) & 1, g, wait_code<6>());
      __syncwarp();
      tc_fence_after_sync();
      const uint32_t scol = tmem + lrow + ((j & 1) ? Gm::S_COL1 : Gm::S_COL0);
      // raw S, 32 columns per load, all loads in flight before one wait
      constexpr int NC = BK / 32;
      uint32_t sr[NC][32];
#pragma unroll
      for (int c = 0; c < NC; ++c) tmem_ld32(scol + c * 32, sr[c]);
      tmem_ld_wait(sr[0]);
#pragma unroll
      for (int c = 1; c < NC; ++c) reg_fence(sr[c]);
      // S is in registers: the S warp may compute tile j+2 into this buffer
      tc_fence_before_sync();
      mbar_arrive(smem_u32(&bar_sfree[j & 1]));
      const int k0 = (j0 + jt) * BK;
      const bool need_mask = (CAUSAL && (k0 + BK - 1 > q0 + p.off)) || (k0 + BK > p.Lk);
      if (need_mask) {
#pragma unroll
        for (int i = 0; i < BK; ++i)
          if (k0 + i > lim) sr[i >> 5][i & 31] = __float_as_uint(-INFINITY);
      }
      // row maximum of the raw scores (scale_log2 > 0 commutes with max):
      // eight independent chains of three-input maxima
      float mx[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) mx[i] = __uint_as_float(sr[0][i]);
#pragma unroll
      for (int e = 8; e < BK; e += 2)
        mx[(e >> 1) & 7] = fmax3(mx[(e >> 1) & 7], __uint_as_float(sr[e >> 5][e & 31]),
                                 __uint_as_float(sr[(e + 1) >> 5][(e + 1) & 31]));
      const float mt = fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7])) * sl2;
      const float m_new = fmaxf(m, mt);
      // Lazy rescaling: the row keeps its reference maximum m until a tile
      // raises the row maximum by more than TAU = 8 (log2 units), so P <= 2^8 and
      // O and l are rescaled only on those (rare) tiles.  O holds P V up to
      // the previous key tile once that MMA is done (none on the first tile:
      // its P V overwrites O).  (Each P V barrier completes once per two
      // tiles and is waited for in order below, so a parity wait cannot
      // mistake an older phase for this one.)
      if (__any_sync(0xffffffffu, m_new > m + Gm::TAU)) {
        const float alpha = ex2_approx(m - m_new);  // 0 while m = -inf
        m = m_new;
        l *= alpha;
        if (j > 0) {
          mbar_wait(smem_u32(&bar_pvdone[(j - 1) & 1]), ((j - 1) >> 1) & 1, g, wait_code<7>());
          __syncwarp();
          tc_fence_after_sync();
#pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            uint32_t rr[32];
            tmem_ld32(tmem + lrow + Gm::O_COL + c * 32, rr);
            tmem_ld_wait(rr);
#pragma unroll
            for (int i = 0; i < 32; ++i) rr[i] = __float_as_uint(__uint_as_float(rr[i]) * alpha);
            tmem_st32(tmem + lrow + Gm::O_COL + c * 32, rr);
          }
        }
      }
      // (decode, block mask: a row that has seen no key keeps m = -inf, P = 0)
      const float mu = ((DECODE || MASKED) && m == -INFINITY) ? 0.f : m;
      // P = exp2(S * scale_log2 - mu), two elements per packed instruction
      const uint64_t sl2x2 = f2_pack(sl2, sl2), nm2 = f2_pack(-mu, -mu);
      uint64_t sum2[2] = {f2_pack(0.f, 0.f), f2_pack(0.f, 0.f)};
      const uint32_t pcol = tmem + lrow + ((j & 1) ? Gm::P_COL1 : Gm::P_COL0);
      // P V of tile j-2 has read this P buffer
      if (j >= 2) {
        mbar_wait(smem_u32(&bar_pvdone[j & 1]), ((j - 2) >> 1) & 1, g, wait_code<29>());
        __syncwarp();
        tc_fence_after_sync();
      }
#pragma unroll
      for (int c = 0; c < NC; ++c) {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          float x0, x1;
          f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[c][2 * i]), __uint_as_float(sr[c][2 * i + 1])), sl2x2, nm2), x0,
                    x1);
          const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
          sum2[c & 1] = f2_add(sum2[c & 1], f2_pack(p0, p1));
          pk[i] = E::pack(p0, p1);
        }
        tmem_st16(pcol + c * 16, pk);
      }
      {
        float s0, s1, s2, s3;
        f2_unpack(sum2[0], s0, s1);
        f2_unpack(sum2[1], s2, s3);
        l += (s0 + s1) + (s2 + s3);
      }
      tmem_st_wait();
      tc_fence_before_sync();
      mbar_arrive(smem_u32(&bar_pready[j & 1]));
    }
    // ---------------- epilogue ----------------
    if (nk > 0) mbar_wait(smem_u32(&bar_pvdone[(nk - 1) & 1]), ((nk - 1) >> 1) & 1, g, wait_code<8>());
    __syncwarp();
    tc_fence_after_sync();
    if constexpr (DECODE) {
      // partial row (split y, packed row bh * Lq + qi) of the combine input
      const bool empty = !(l > 0.f);
      const float inv_l = empty ? 0.f : 1.f / l;
      const size_t x = (static_cast<size_t>(blockIdx.y) * gridDim.x + bh) * p.Lq + qi;
      const size_t n_ws_rows = static_cast<size_t>(gridDim.y) * gridDim.x * p.Lq;  // splits x packed rows
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t rr[32];
        tmem_ld32(tmem + lrow + Gm::O_COL + c * 32, rr);
        tmem_ld_wait(rr);
        if (qi < p.Lq && dbg_in_range(x * D + c * 32, 32, n_ws_rows * D, p.status, 3))
          store_row32_f32(p.ws + x * D + c * 32, rr, inv_l);
      }
      if (qi < p.Lq && dbg_in_range(x, 1, n_ws_rows, p.status, 4)) p.ws_lse[x] = empty ? -INFINITY : m + log2f(l);
    } else {
      const bool empty = MASKED && !(l > 0.f);  // the row saw no key: O = 0, lse = +inf
      const float inv_l = empty ? 0.f : 1.f / l;
      typename E::T* orow = reinterpret_cast<typename E::T*>(p.o) + (static_cast<size_t>(bh) * p.Lq + qi) * D;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t rr[32];
        if (!MASKED || nk > 0) {  // the same for the whole CTA: tcgen05.ld is warp-collective
          tmem_ld32(tmem + lrow + Gm::O_COL + c * 32, rr);
          tmem_ld_wait(rr);
        }
        if (empty) {  // (also every row when no key tile is kept)
#pragma unroll
          for (int i = 0; i < 32; ++i) rr[i] = 0u;
        }
        if (qi < p.Lq && dbg_in_range((static_cast<size_t>(bh) * p.Lq + qi) * D + c * 32, 32, n_qrows * D, p.status, 5))
          store_row32<BF16>(orow + c * 32, rr, inv_l);
      }
      if (qi < p.Lq && dbg_in_range(static_cast<size_t>(bh) * p.Lq + qi, 1, n_qrows, p.status, 6))
        p.lse[static_cast<size_t>(bh) * p.Lq + qi] = empty ? INFINITY : m + log2f(l);
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
