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
// Warp roles (320 threads per CTA): warps 0-7 row threads -- warp w owns
// TMEM lanes 32*(w%4)..+31 (key rows) and query columns 32*(w/4)..+31 of
// each tile, and loads the lse / delta values of its queries itself;
// warp 8 producer (TMA for the Q and dO rings); warp 9 MMA issuer and TMEM
// owner.
#pragma once

#include "kernel_common.cuh"

namespace gbattn {

// P^T of one query tile handed from the dV CTA to the dK CTA of a cluster:
// 128 key rows x 64 queries of 16-bit values, as eight 2 KB blocks, one per
// row warp (warp w = 4 * half + quad holds key rows 32 * quad .. +31 and
// queries 32 * half .. +31 in both CTAs), so each warp sends its own block
// with one bulk copy.  In a block, lane l's 64 bytes (four 16-byte chunks of
// eight queries) start at 64 l, chunk c stored at position c ^ ((l >> 1) & 3)
// so that eight consecutive lanes cover all banks.  Two slots: the dV CTA may
// run one query tile ahead.
struct PtXch {
  static constexpr int SLOT_BYTES = 128 * 128;
  static constexpr int BLOCK_BYTES = 32 * 64;
  static constexpr int SLOTS = 2;
  static constexpr int BYTES = SLOTS * SLOT_BYTES;
  __device__ __forceinline__ static uint32_t block(uint32_t base, int slot, int warp) {
    return base + slot * SLOT_BYTES + warp * BLOCK_BYTES;
  }
  __device__ __forceinline__ static uint32_t addr(uint32_t base, int slot, int warp, int lane, int chunk) {
    return block(base, slot, warp) + lane * 64 + ((chunk ^ ((lane >> 1) & 3)) << 4);
  }
};

// mbarriers of the hand-off, in the shared memory of both CTAs (the kernel
// declares them, so they sit at the same offset in either CTA).  pfull, in
// the dK CTA: one local arrival that expects the slot's bytes, which the dV
// CTA's bulk copies complete (the bytes are visible to a thread that sees the
// phase complete, as for a TMA load).  pfree, in the dV CTA: one
// arrival per warp of the dK CTA's row threads once they have used the
// slot's values.
struct PtXchBars {
  uint64_t pfull[PtXch::SLOTS], pfree[PtXch::SLOTS];
};

// Q and dO tiles of 64 queries x 256 columns (four 64-column chunks, 32 KB)
// sit in two rings of their own, each slot freed by the MMA that last reads
// it: the slot a tile is loaded into is then free one or two query tiles
// before that tile is needed, which covers the TMA's latency.  The per-query
// lse / delta values are loaded by the row threads themselves (one value per
// lane, a query tile ahead) and spread with shuffles.
__device__ __forceinline__ void load_tile256(uint32_t dst, const CUtensorMap* map, uint32_t bar, int q0, int zq) {
#pragma unroll
  for (int c = 0; c < 4; ++c) tma_load_3d_w(dst + c * 64 * 128, map, bar, c * 64, q0, zq);
}

// D = 256, dK half (cluster rank 1).  V sits in tensor memory as the A
// operand of dP^T = V dO^T (copied in by the row threads), so only the dO
// tile is read from shared memory; P^T comes from the partner CTA.  Tensor
// memory: dK (256 columns), V (128: 256 16-bit values per row), dP^T (two
// buffers of 64).  The row threads write dS^T (16-bit pairs) over the dP^T
// columns they have read, and the MMA warp issues dK += dS^T Q, then dP^T of
// the tile after next into the same buffer (tcgen05 MMAs of one thread run
// in issue order).
struct Dk256Geom {
  static constexpr int D = 256, BK = 128, BQ = 64, NCH = 4;
  static constexpr int Q_BYTES = NCH * BQ * 128;  // one Q or dO tile, 32 KB
  static constexpr int NQ = 3, NO = 3;            // Q and dO ring slots
  static constexpr int XCH_OFF = (NQ + NO) * Q_BYTES;  // from the 1024-aligned base
  static constexpr int SMEM_BYTES = 1024 + XCH_OFF + PtXch::BYTES;
  static constexpr int DK_COL = 0, V_COL = 256, DPT_COL = 384;  // dP^T: 2 x 64
  static constexpr int TMEM_COLS = 512;
  static constexpr int NUM_COMPUTE_WARPS = 8;
  static constexpr int NCT = 32 * NUM_COMPUTE_WARPS;
  static constexpr int PRODUCER_WARP = NUM_COMPUTE_WARPS;
  static constexpr int MMA_WARP = NUM_COMPUTE_WARPS + 1;
  static constexpr int NUM_THREADS = 32 * (NUM_COMPUTE_WARPS + 2);
  static_assert(SMEM_BYTES + 1024 <= kMaxDynSmem, "shared memory budget (1 KB left for static variables)");
  static_assert(NO >= 3, "dP^T runs two query tiles ahead of dK");
  static_assert(DPT_COL + 2 * BQ <= TMEM_COLS, "tensor memory budget");
};

template <bool BF16, bool CAUSAL, bool MASKED>
__device__ __forceinline__ void dk256_tile(const CUtensorMap& tmQ, const CUtensorMap& tmdO, const BwdParams& p,
                                           const int bhk, const int kt, PtXchBars& xb) {
  using Gm = Dk256Geom;
  using E = Elem<BF16>;
  constexpr int D = Gm::D, BQ = Gm::BQ, BK = Gm::BK, NQ = Gm::NQ, NO = Gm::NO, NCT = Gm::NCT;

  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t bar_vready, bar_qfull[NQ], bar_qempty[NQ], bar_ofull[NO], bar_oempty[NO], bar_dpfull[2],
      bar_dsready[2], bar_accdone;
  __shared__ uint32_t tmem_slot;
  __shared__ volatile int abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t sQ0 = sbase;
  const uint32_t sdO0 = sQ0 + NQ * Gm::Q_BYTES;
  const uint32_t sX = sbase + Gm::XCH_OFF;

  const int b = bhk / p.Hkv, hk = bhk - b * p.Hkv;
  const int k0 = kt * BK;
  const int qt_start = CAUSAL ? max(0, k0 - p.off) / BQ : 0;
  // query tile qt is computed (block mask: the CTA's 128 keys are one mask
  // column, a 64-row query tile half a mask row)
  auto keep = [&](int qt) { return !MASKED || mask_keep(p, qt >> 1, kt); };
  const int n_iter = p.G * count_kept<MASKED>(keep, qt_start, p.n_qtiles);  // (query head, query tile) iterations
  const WaitGuard g{&abort_flag, p.status, p.limit_ns};
  // extents for the debug build's index checks: rows of q / dq / lse /
  // delta, of dk / dv, and of the k / v buffers (pitch kv_pitch per head)
  [[maybe_unused]] const size_t n_qrows = static_cast<size_t>(p.B) * p.Hq * p.Lq;
  [[maybe_unused]] const size_t n_krows = static_cast<size_t>(p.B) * p.Hkv * p.Lk;
  [[maybe_unused]] const size_t n_kvbuf = (static_cast<size_t>(p.B) * p.Hkv - 1) * p.kv_pitch + p.Lk;

  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(smem_u32(&bar_vready), NCT);
    for (int s = 0; s < NQ; ++s) {
      mbar_init(smem_u32(&bar_qfull[s]), 1);   // TMA expect_tx arrive
      mbar_init(smem_u32(&bar_qempty[s]), 1);  // dK's commit
    }
    for (int s = 0; s < NO; ++s) {
      mbar_init(smem_u32(&bar_ofull[s]), 1);
      mbar_init(smem_u32(&bar_oempty[s]), 1);  // dP^T's commit
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
  auto qw = kept_walk<MASKED>(keep, p.n_qtiles);

  if (warp == Gm::PRODUCER_WARP) {
    // ---------------- producer (whole warp) ----------------
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmdO);
    }
    __syncwarp();
    RingPos<NQ> rq;
    RingPos<NO> ro;
    // the Q and dO loads walk the (head, query tile) list separately: a
    // walker carries state under a mask
    auto wq = qw, wo = qw;
    int gq = 0, tq = wq.first(qt_start);  // query head in the group and query tile of the next Q load
    int go = 0, to = wo.first(qt_start);  // and of the next dO load
    // Q and dO tiles issued; after an abort (a wait ran out) no further copy
    // is issued, so the drains below cover every copy still in flight
    int nqi = 0, noi = 0;
    auto load_q = [&](int i) {
      if (i >= NQ) mbar_wait(smem_u32(&bar_qempty[rq.slot]), rq.phase ^ 1u, g, wait_code<20>());
      __syncwarp();
      if (abort_flag) return false;
      ++nqi;
      const uint32_t bar = smem_u32(&bar_qfull[rq.slot]);
      mbar_arrive_expect_tx_w(bar, Gm::Q_BYTES);
      load_tile256(sQ0 + rq.slot * Gm::Q_BYTES, &tmQ, bar, tq * BQ, b * p.Hq + hk * p.G + gq);
      rq.next();
      tq = wq.next(tq);
      if (tq >= p.n_qtiles) tq = wq.first(qt_start), ++gq;
      return true;
    };
    auto load_o = [&](int i) {
      if (i >= NO) mbar_wait(smem_u32(&bar_oempty[ro.slot]), ro.phase ^ 1u, g, wait_code<28>());
      __syncwarp();
      if (abort_flag) return false;
      ++noi;
      const uint32_t bar = smem_u32(&bar_ofull[ro.slot]);
      mbar_arrive_expect_tx_w(bar, Gm::Q_BYTES);
      load_tile256(sdO0 + ro.slot * Gm::Q_BYTES, &tmdO, bar, to * BQ, b * p.Hq + hk * p.G + go);
      ro.next();
      to = wo.next(to);
      if (to >= p.n_qtiles) to = wo.first(qt_start), ++go;
      return true;
    };
    // in the order the MMA warp needs them: dO runs two query tiles ahead of Q
    for (int i = 0; i < 2 && i < n_iter; ++i)
      if (!load_o(i)) break;
    for (int it = 0; it < n_iter && !abort_flag; ++it) {
      if (!load_q(it)) break;
      if (it + 2 < n_iter && !load_o(it + 2)) break;
    }
    // the last Q and dO copies issued (a slot is refilled only after its
    // release, so each slot has at most one copy in flight)
    for (int i = (nqi > NQ ? nqi - NQ : 0); i < nqi; ++i)
      mbar_wait_drain(smem_u32(&bar_qfull[i % NQ]), (i / NQ) & 1);
    for (int i = (noi > NO ? noi - NO : 0); i < noi; ++i)
      mbar_wait_drain(smem_u32(&bar_ofull[i % NO]), (i / NO) & 1);
  } else if (warp == Gm::MMA_WARP) {
    // ---------------- MMA issuer ----------------
    constexpr uint32_t IDESC_DP = make_idesc_f16(128, BQ, BF16, false, false);
    constexpr uint32_t IDESC_ACC = make_idesc_f16(128, D, BF16, false, true);
    const uint64_t dOk = make_sdesc_sw128(sdO0, 16, 1024);       // dO slot 0, K-major
    const uint64_t dQm = make_sdesc_sw128(sQ0, BQ * 128, 1024);  // Q slot 0, MN-major
    RingPos<NQ> rq;
    RingPos<NO> ro;
    // dP^T(it) = V dO^T into buffer it & 1 (V from tensor memory)
    auto issue_dp = [&](int it) {
      mbar_wait(smem_u32(&bar_ofull[ro.slot]), ro.phase, g, wait_code<22>());
      __syncwarp();
      tc_fence_after_sync();
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t qo = ro.slot * Gm::Q_BYTES + (kk >> 2) * (BQ * 128) + (kk & 3) * 32;
        mma_ts_w(tmem + Gm::DPT_COL + (it & 1) * BQ, tmem + Gm::V_COL + kk * 8, sdesc_add(dOk, qo), IDESC_DP,
                 kk > 0 ? 1u : 0u);
      }
      mma_commit_w(smem_u32(&bar_dpfull[it & 1]));
      mma_commit_w(smem_u32(&bar_oempty[ro.slot]));
      ro.next();
    };
    mbar_wait(smem_u32(&bar_vready), 0, g, wait_code<21>());
    for (int it = 0; it < 2 && it < n_iter; ++it) issue_dp(it);
    for (int it = 0; it < n_iter; ++it) {
      const int buf = it & 1;
      // dS^T(it) is in dP^T buffer buf
      mbar_wait(smem_u32(&bar_dsready[buf]), (it >> 1) & 1, g, wait_code<23>());
      mbar_wait(smem_u32(&bar_qfull[rq.slot]), rq.phase, g, wait_code<24>());
      __syncwarp();
      tc_fence_after_sync();
      // A operand: queries 32h..32h+31 of warpgroup h as pairs in columns
      // 32h..32h+15 of the buffer
#pragma unroll
      for (int kk = 0; kk < BQ / 16; ++kk) {
        const uint32_t acol = Gm::DPT_COL + buf * BQ + (kk >> 1) * 32 + (kk & 1) * 8;
        mma_ts_w(tmem + Gm::DK_COL, tmem + acol, sdesc_add(dQm, rq.slot * Gm::Q_BYTES + kk * 2048), IDESC_ACC,
                 (it > 0 || kk > 0) ? 1u : 0u);
      }
      mma_commit_w(smem_u32(&bar_qempty[rq.slot]));
      rq.next();
      // dP^T(it+2) overwrites dS^T(it) behind the dK MMAs that read it
      if (it + 2 < n_iter) issue_dp(it + 2);
    }
    mma_commit_w(smem_u32(&bar_accdone));
    mbar_wait_drain(smem_u32(&bar_accdone), 0);
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
          if (kj < p.Lk && dbg_in_range((static_cast<size_t>(bhk) * p.kv_pitch + kj) * D + half * 128 + 8 * (c * 4 + v),
                                        8, n_kvbuf * D, p.status, 19))
            x = src[c * 4 + v];
          t16[4 * v + 0] = x.x, t16[4 * v + 1] = x.y, t16[4 * v + 2] = x.z, t16[4 * v + 3] = x.w;
        }
        tmem_st16(tmem + lrow + Gm::V_COL + half * 64 + c * 16, t16);
      }
      tmem_st_wait();
      tc_fence_before_sync();
      mbar_arrive(smem_u32(&bar_vready));
    }
    // delta of query half*32 + lane of a query tile (0 past Lq)
    auto delta_of = [&](int qt, int gq) {
      const int qi = qt * BQ + half * 32 + lane;
      const size_t row = static_cast<size_t>(b * p.Hq + hk * p.G + gq) * p.Lq + qi;
      return qi < p.Lq && dbg_in_range(row, 1, n_qrows, p.status, 20) ? p.delta[row] : 0.f;
    };
    int gi = 0, qtile = qw.first(qt_start);
    float dl = n_iter > 0 ? delta_of(qtile, gi) : 0.f;
    for (int it = 0; it < n_iter; ++it) {
      const int buf = it & 1;
      const float dl_cur = dl;
      qtile = qw.next(qtile);
      if (qtile >= p.n_qtiles) qtile = qw.first(qt_start), ++gi;
      if (it + 1 < n_iter) dl = delta_of(qtile, gi);  // next query tile's, in flight during this one
      mbar_wait(smem_u32(&bar_dpfull[buf]), (it >> 1) & 1, g, wait_code<25>());
      __syncwarp();
      tc_fence_after_sync();
      const uint32_t dcol = tmem + lrow + Gm::DPT_COL + buf * BQ + half * 32;
      uint32_t dr[32];
      tmem_ld32(dcol, dr);
      // P^T(it) from the dV CTA: 32 queries (four chunks) of this thread's key row
      mbar_wait(smem_u32(&xb.pfull[buf]), (it >> 1) & 1, g, wait_code<26>());
      // the slot's next use (query tile it + 2) expects its bytes: the dV CTA
      // cannot write them before every warp here has released this use
      if (threadIdx.x == 0 && it + 2 < n_iter && !abort_flag)
        mbar_arrive_expect_tx(smem_u32(&xb.pfull[buf]), PtXch::SLOT_BYTES);
      uint4 pv[4];
#pragma unroll
      for (int v = 0; v < 4; ++v) pv[v] = ld_shared_v4(PtXch::addr(sX, buf, warp, lane, v));
      tmem_ld_wait(dr);
      const uint32_t pw[16] = {pv[0].x, pv[0].y, pv[0].z, pv[0].w, pv[1].x, pv[1].y, pv[1].z, pv[1].w,
                               pv[2].x, pv[2].y, pv[2].z, pv[2].w, pv[3].x, pv[3].y, pv[3].z, pv[3].w};
      uint32_t dk[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int c0 = 2 * i;
        const float2 pp = E::unpack(pw[i]);
        const uint64_t dl2 = f2_pack(__shfl_sync(0xffffffffu, dl_cur, c0), __shfl_sync(0xffffffffu, dl_cur, c0 + 1));
        const uint64_t d2 = f2_sub(f2_pack(__uint_as_float(dr[c0]), __uint_as_float(dr[c0 + 1])), dl2);
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
    mbar_wait(smem_u32(&bar_accdone), 0, g, wait_code<27>());
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
      if (kj < p.Lk && dbg_in_range((static_cast<size_t>(bhk) * p.Lk + kj) * D + c * 32, 32, n_krows * D, p.status, 21))
        store_row32<BF16>(dst + c * 32, rr, p.scale);
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == Gm::MMA_WARP) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, Gm::TMEM_COLS);
  }
  // The last two hand-offs have landed before this CTA meets its partner
  // at the final cluster barrier (after which either may exit): at once in
  // a normal run, where every one of them was waited for; after an abort
  // the partner may have sent part of a slot, and the bounded drain outlasts
  // any copy still landing.
  if (threadIdx.x == 0)
    for (int it = (n_iter > PtXch::SLOTS ? n_iter - PtXch::SLOTS : 0); it < n_iter; ++it)
      mbar_wait_drain(smem_u32(&xb.pfull[it & 1]), (it >> 1) & 1);
}

// D = 256, dV half (cluster rank 0): K in tensor memory as the A operand of
// S^T = K Q^T (copied in by the row threads), so shared memory holds only the
// Q and dO rings.  Tensor memory: dV (256 columns), K (128), S^T (two buffers
// of 64).  The row threads turn S^T into P^T (16-bit pairs) and write it over
// the columns they read and into a local staging slot, which each warp sends
// to the partner CTA with one bulk copy of its block (so no thread waits on
// remote stores); the MMA warp issues dV += P^T dO, then S^T of the tile
// after next into the same buffer.  A quarter of the exponentials use a
// polynomial on the FMA pipe: with only the P^T work left on these row
// threads, the MUFU unit would otherwise set their pace (the share was
// measured: 4 of 16 pairs beat 0, 2, 3, 5, 6, 8, 12 and 16).
struct Dv256Geom {
  static constexpr int D = 256, BK = 128, BQ = 64, NCH = 4;
  static constexpr int Q_BYTES = NCH * BQ * 128;  // one Q or dO tile, 32 KB
  static constexpr int NQ = 3, NO = 3;            // Q and dO ring slots
  static constexpr int STAGE_OFF = (NQ + NO) * Q_BYTES;  // P^T staging slots (the hand-off layout)
  static constexpr int SMEM_BYTES = 1024 + STAGE_OFF + PtXch::BYTES;
  // element pairs (of 16 per thread and query tile) whose exponentials use
  // the polynomial on the FMA pipe instead of the MUFU unit
#ifndef GBATTN_DV256_POLY
  static constexpr int POLY = 4;
#else
  static constexpr int POLY = GBATTN_DV256_POLY;
#endif
  static_assert(POLY >= 0 && POLY <= 16, "polynomial share");
  static_assert(SMEM_BYTES + 1024 <= kMaxDynSmem, "shared memory budget (1 KB left for static variables)");
  static constexpr int DV_COL = 0, K_COL = 256, ST_COL = 384;  // S^T: 2 x 64
  static constexpr int TMEM_COLS = 512;
  static constexpr int NUM_COMPUTE_WARPS = 8;
  static constexpr int NCT = 32 * NUM_COMPUTE_WARPS;
  static constexpr int PRODUCER_WARP = NUM_COMPUTE_WARPS;
  static constexpr int MMA_WARP = NUM_COMPUTE_WARPS + 1;
  static constexpr int NUM_THREADS = 32 * (NUM_COMPUTE_WARPS + 2);
  static_assert(NQ >= 3, "S^T runs two query tiles ahead of dV");
  static_assert(ST_COL + 2 * BQ <= TMEM_COLS, "tensor memory budget");
};

template <bool BF16, bool CAUSAL, bool MASKED>
__device__ __forceinline__ void dv256_tile(const CUtensorMap& tmQ, const CUtensorMap& tmdO, const BwdParams& p,
                                           const int bhk, const int kt, PtXchBars& xb) {
  using Gm = Dv256Geom;
  using E = Elem<BF16>;
  constexpr int D = Gm::D, BQ = Gm::BQ, BK = Gm::BK, NQ = Gm::NQ, NO = Gm::NO, NCT = Gm::NCT;

  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t bar_kready, bar_qfull[NQ], bar_qempty[NQ], bar_ofull[NO], bar_oempty[NO], bar_sfull[2],
      bar_pready[2], bar_accdone;
  __shared__ uint32_t tmem_slot;
  __shared__ volatile int abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t sQ0 = sbase;
  const uint32_t sdO0 = sQ0 + NQ * Gm::Q_BYTES;
  const uint32_t sStage = sbase + Gm::STAGE_OFF;                   // P^T staging slots
  const uint32_t sX1 = cluster_map(sbase + Dk256Geom::XCH_OFF, 1);  // the dK CTA's hand-off slots

  const int b = bhk / p.Hkv, hk = bhk - b * p.Hkv;
  const int k0 = kt * BK;
  const int qt_start = CAUSAL ? max(0, k0 - p.off) / BQ : 0;
  // query tile qt is computed (block mask: the CTA's 128 keys are one mask
  // column, a 64-row query tile half a mask row)
  auto keep = [&](int qt) { return !MASKED || mask_keep(p, qt >> 1, kt); };
  const int n_iter = p.G * count_kept<MASKED>(keep, qt_start, p.n_qtiles);  // (query head, query tile) iterations
  const WaitGuard g{&abort_flag, p.status, p.limit_ns};
  // extents for the debug build's index checks: rows of q / dq / lse /
  // delta, of dk / dv, and of the k / v buffers (pitch kv_pitch per head)
  [[maybe_unused]] const size_t n_qrows = static_cast<size_t>(p.B) * p.Hq * p.Lq;
  [[maybe_unused]] const size_t n_krows = static_cast<size_t>(p.B) * p.Hkv * p.Lk;
  [[maybe_unused]] const size_t n_kvbuf = (static_cast<size_t>(p.B) * p.Hkv - 1) * p.kv_pitch + p.Lk;

  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(smem_u32(&bar_kready), NCT);
    for (int s = 0; s < NQ; ++s) {
      mbar_init(smem_u32(&bar_qfull[s]), 1);   // TMA expect_tx arrive
      mbar_init(smem_u32(&bar_qempty[s]), 1);  // S^T's commit
    }
    for (int s = 0; s < NO; ++s) {
      mbar_init(smem_u32(&bar_ofull[s]), 1);
      mbar_init(smem_u32(&bar_oempty[s]), 1);  // dV's commit
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
  auto qw = kept_walk<MASKED>(keep, p.n_qtiles);

  if (warp == Gm::PRODUCER_WARP) {
    // ---------------- producer (whole warp) ----------------
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmdO);
    }
    __syncwarp();
    RingPos<NQ> rq;
    RingPos<NO> ro;
    // the Q and dO loads walk the (head, query tile) list separately: a
    // walker carries state under a mask
    auto wq = qw, wo = qw;
    int gq = 0, tq = wq.first(qt_start);  // query head in the group and query tile of the next Q load
    int go = 0, to = wo.first(qt_start);  // and of the next dO load
    // Q and dO tiles issued; after an abort (a wait ran out) no further copy
    // is issued, so the drains below cover every copy still in flight
    int nqi = 0, noi = 0;
    auto load_q = [&](int i) {
      if (i >= NQ) mbar_wait(smem_u32(&bar_qempty[rq.slot]), rq.phase ^ 1u, g, wait_code<45>());
      __syncwarp();
      if (abort_flag) return false;
      ++nqi;
      const uint32_t bar = smem_u32(&bar_qfull[rq.slot]);
      mbar_arrive_expect_tx_w(bar, Gm::Q_BYTES);
      load_tile256(sQ0 + rq.slot * Gm::Q_BYTES, &tmQ, bar, tq * BQ, b * p.Hq + hk * p.G + gq);
      rq.next();
      tq = wq.next(tq);
      if (tq >= p.n_qtiles) tq = wq.first(qt_start), ++gq;
      return true;
    };
    auto load_o = [&](int i) {
      if (i >= NO) mbar_wait(smem_u32(&bar_oempty[ro.slot]), ro.phase ^ 1u, g, wait_code<57>());
      __syncwarp();
      if (abort_flag) return false;
      ++noi;
      const uint32_t bar = smem_u32(&bar_ofull[ro.slot]);
      mbar_arrive_expect_tx_w(bar, Gm::Q_BYTES);
      load_tile256(sdO0 + ro.slot * Gm::Q_BYTES, &tmdO, bar, to * BQ, b * p.Hq + hk * p.G + go);
      ro.next();
      to = wo.next(to);
      if (to >= p.n_qtiles) to = wo.first(qt_start), ++go;
      return true;
    };
    // in the order the MMA warp needs them: Q runs two query tiles ahead of dO
    for (int i = 0; i < 2 && i < n_iter; ++i)
      if (!load_q(i)) break;
    for (int it = 0; it < n_iter && !abort_flag; ++it) {
      if (!load_o(it)) break;
      if (it + 2 < n_iter && !load_q(it + 2)) break;
    }
    // the last Q and dO copies issued (a slot is refilled only after its
    // release, so each slot has at most one copy in flight)
    for (int i = (nqi > NQ ? nqi - NQ : 0); i < nqi; ++i)
      mbar_wait_drain(smem_u32(&bar_qfull[i % NQ]), (i / NQ) & 1);
    for (int i = (noi > NO ? noi - NO : 0); i < noi; ++i)
      mbar_wait_drain(smem_u32(&bar_ofull[i % NO]), (i / NO) & 1);
  } else if (warp == Gm::MMA_WARP) {
    // ---------------- MMA issuer ----------------
    constexpr uint32_t IDESC_S = make_idesc_f16(128, BQ, BF16, false, false);
    constexpr uint32_t IDESC_ACC = make_idesc_f16(128, D, BF16, false, true);
    const uint64_t dQk = make_sdesc_sw128(sQ0, 16, 1024);         // Q slot 0, K-major
    const uint64_t dOm = make_sdesc_sw128(sdO0, BQ * 128, 1024);  // dO slot 0, MN-major
    RingPos<NQ> rq;
    RingPos<NO> ro;
    // S^T(it) = K Q^T into buffer it & 1 (K from tensor memory)
    auto issue_s = [&](int it) {
      mbar_wait(smem_u32(&bar_qfull[rq.slot]), rq.phase, g, wait_code<46>());
      __syncwarp();
      tc_fence_after_sync();
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t qo = rq.slot * Gm::Q_BYTES + (kk >> 2) * (BQ * 128) + (kk & 3) * 32;
        mma_ts_w(tmem + Gm::ST_COL + (it & 1) * BQ, tmem + Gm::K_COL + kk * 8, sdesc_add(dQk, qo), IDESC_S,
                 kk > 0 ? 1u : 0u);
      }
      mma_commit_w(smem_u32(&bar_sfull[it & 1]));
      mma_commit_w(smem_u32(&bar_qempty[rq.slot]));
      rq.next();
    };
    mbar_wait(smem_u32(&bar_kready), 0, g, wait_code<47>());
    for (int it = 0; it < 2 && it < n_iter; ++it) issue_s(it);
    for (int it = 0; it < n_iter; ++it) {
      const int buf = it & 1;
      mbar_wait(smem_u32(&bar_pready[buf]), (it >> 1) & 1, g, wait_code<48>());
      mbar_wait(smem_u32(&bar_ofull[ro.slot]), ro.phase, g, wait_code<49>());
      __syncwarp();
      tc_fence_after_sync();
      // A operand: queries 32h..32h+31 of warpgroup h as pairs in columns
      // 32h..32h+15 of the buffer
#pragma unroll
      for (int kk = 0; kk < BQ / 16; ++kk) {
        const uint32_t acol = Gm::ST_COL + buf * BQ + (kk >> 1) * 32 + (kk & 1) * 8;
        mma_ts_w(tmem + Gm::DV_COL, tmem + acol, sdesc_add(dOm, ro.slot * Gm::Q_BYTES + kk * 2048), IDESC_ACC,
                 (it > 0 || kk > 0) ? 1u : 0u);
      }
      mma_commit_w(smem_u32(&bar_oempty[ro.slot]));
      ro.next();
      // S^T(it+2) overwrites P^T(it) behind the dV MMAs that read it
      if (it + 2 < n_iter) issue_s(it + 2);
    }
    mma_commit_w(smem_u32(&bar_accdone));
    mbar_wait_drain(smem_u32(&bar_accdone), 0);
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
    {
      const uint4* src = reinterpret_cast<const uint4*>(reinterpret_cast<const typename E::T*>(p.k) +
                                                        (static_cast<size_t>(bhk) * p.kv_pitch + kj) * D + half * 128);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t t16[16];
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          uint4 x = make_uint4(0u, 0u, 0u, 0u);
          if (kj < p.Lk && dbg_in_range((static_cast<size_t>(bhk) * p.kv_pitch + kj) * D + half * 128 + 8 * (c * 4 + v),
                                        8, n_kvbuf * D, p.status, 22))
            x = src[c * 4 + v];
          t16[4 * v + 0] = x.x, t16[4 * v + 1] = x.y, t16[4 * v + 2] = x.z, t16[4 * v + 3] = x.w;
        }
        tmem_st16(tmem + lrow + Gm::K_COL + half * 64 + c * 16, t16);
      }
      tmem_st_wait();
      tc_fence_before_sync();
      mbar_arrive(smem_u32(&bar_kready));
    }
    // -lse of query half*32 + lane of a query tile (-inf past Lq)
    auto nlse_of = [&](int qt, int gq) {
      const int qi = qt * BQ + half * 32 + lane;
      const size_t row = static_cast<size_t>(b * p.Hq + hk * p.G + gq) * p.Lq + qi;
      return qi < p.Lq && dbg_in_range(row, 1, n_qrows, p.status, 23) ? -p.lse[row] : -INFINITY;
    };
    int gi = 0, qtile = qw.first(qt_start);
    float nl = n_iter > 0 ? nlse_of(qtile, gi) : 0.f;
    for (int it = 0; it < n_iter; ++it) {
      const int buf = it & 1;
      const int q0 = qtile * BQ;
      const float nl_cur = nl;
      qtile = qw.next(qtile);
      if (qtile >= p.n_qtiles) qtile = qw.first(qt_start), ++gi;
      if (it + 1 < n_iter) nl = nlse_of(qtile, gi);  // next query tile's, in flight during this one
      mbar_wait(smem_u32(&bar_sfull[buf]), (it >> 1) & 1, g, wait_code<50>());
      __syncwarp();
      tc_fence_after_sync();
      const uint32_t scol = tmem + lrow + Gm::ST_COL + buf * BQ + half * 32;
      uint32_t sr[32];
      tmem_ld32(scol, sr);
      tmem_ld_wait(sr);
      const bool need_mask = CAUSAL && (q0 < k0 + BK - 1 - p.off);
      const int qc0 = q0 + half * 32;
      uint32_t pk[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int c0 = 2 * i;
        float x0, x1, p0, p1;
        const uint64_t nl2 = f2_pack(__shfl_sync(0xffffffffu, nl_cur, c0), __shfl_sync(0xffffffffu, nl_cur, c0 + 1));
        f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[c0]), __uint_as_float(sr[c0 + 1])), sl2x2, nl2), x0, x1);
        if ((i + 1) * Gm::POLY / 16 > i * Gm::POLY / 16) {  // POLY of the 16 pairs, spread evenly
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
      }
      tmem_st16(scol, pk);
      // P^T(it) into this warp's block of staging slot buf, once the dK CTA
      // has used the slot's previous contents (so their copy has completed
      // too), then to the dK CTA's slot with one bulk copy per warp,
      // completing on its pfull (the proxy fence makes the stores visible to
      // the copy)
      if (it >= 2) mbar_wait(smem_u32(&xb.pfree[buf]), ((it >> 1) & 1) ^ 1, g, wait_code<56>());
      if (!abort_flag) {  // after an abort nothing more is sent
#pragma unroll
        for (int v = 0; v < 4; ++v)
          st_shared_v4(PtXch::addr(sStage, buf, warp, lane, v), pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
        fence_proxy_async_smem();
        __syncwarp();
        bulk_s2cluster_w(PtXch::block(sX1, buf, warp), PtXch::block(sStage, buf, warp), PtXch::BLOCK_BYTES,
                         cluster_map(smem_u32(&xb.pfull[buf]), 1));
      }
      tmem_st_wait();
      tc_fence_before_sync();
      mbar_arrive(smem_u32(&bar_pready[buf]));
    }
    mbar_wait(smem_u32(&bar_accdone), 0, g, wait_code<55>());
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
      if (kj < p.Lk && dbg_in_range((static_cast<size_t>(bhk) * p.Lk + kj) * D + c * 32, 32, n_krows * D, p.status, 24))
        store_row32<BF16>(dst + c * 32, rr, 1.f);
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
  // A dQ kernel launched behind this one may start filling the SMs this grid
  // frees as soon as every CTA of it is running (it reads none of its outputs).
  if (threadIdx.x == 0) grid_launch_dependents();
  const int bhk = static_cast<int>(blockIdx.x >> 1), kt = static_cast<int>(blockIdx.y);
  if (cluster_ctarank() == 1)
    dk256_tile<BF16, CAUSAL, MASKED>(tmQ, tmdO, p, bhk, kt, xb);
  else
    dv256_tile<BF16, CAUSAL, MASKED>(tmQ, tmdO, p, bhk, kt, xb);
  // neither CTA leaves while the other may still write its shared memory
  cluster_sync_all();
}

}  // namespace gbattn
