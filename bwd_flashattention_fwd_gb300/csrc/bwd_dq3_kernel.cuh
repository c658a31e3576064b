// Backward, dQ kernel for head dims up to 128: same mathematics as
// bwd_dq_kernel.cuh ("feat(attention): complete Flash Attention VJP
// implementation", sections "Background" and "Two-Kernel Design": the dQ
// kernel owns query rows and loops over key tiles; S = Q K^T and dP = dO V^T
// are recomputed, P = exp2(S * scale_log2 - lse), dS = P * (dP - delta),
// dQ += dS K, and dQ is scaled by `scale` at the end).
//
// Shared-memory bandwidth (128 B per clock per SM) is what limits an MMA
// whose two operands both come from shared memory at N = 64.  Q and dO do not
// change over a query tile's key loop, so the row threads copy them into
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
// Persistent: one CTA per SM walks a list of (query tile, head) work items,
// heaviest query tiles first, each CTA taking the next item from a global
// counter when it needs one, so a CTA that starts late (the kernel is
// launched to fill the SMs the dK/dV kernel frees in its last wave) simply
// takes fewer items.  The producer warp takes the items and hands their
// indices to the other warps through a four-slot ring in shared memory.
// While a CTA works on item i, its producer warp prefetches item i+1's Q and
// dO tiles into shared memory with TMA, so starting the next item costs a
// shared-to-tensor-memory copy instead of a global-memory round trip.  Once
// the row threads have copied it out, the same buffer stages the finished
// item's dQ (16-bit, in the swizzled layout of the output's tensor map), and
// the producer writes it out with TMA stores before it loads the next Q and
// dO there: the row threads never wait on a global store.
// Barrier phases count key tiles and items over the CTA's whole life.
//
// Warp roles (352 threads): warps 0-7 row threads -- warp w owns TMEM lanes
// 32*(w%4)..+31 (query rows) and key columns 32*(w/4)..+31 of each 64-key
// tile, and copies D/2 columns of its rows of Q and dO into tensor memory;
// warp 8 TMA producer (Q/dO tiles, and K_j and V_j together into one ring
// stage); warp 9 issues S = Q K^T and owns the TMEM allocation; warp 10
// issues dQ += dS K and dP = dO V^T.  All row warps run one code path (a
// share of exponentials on the FMA pipe, ex2_poly2, can be compiled in with
// GBATTN_DQ_POLY; none is fastest).
//
// MASKED: block-sparse variant ("feat(attention): complete Flash Attention
// VJP implementation", section "Sparse Block Masks": the dQ kernel skips the
// key blocks whose mask entry is zero).  A query tile is one 128-row mask
// block and a key tile half of a 128-key block; skipped key tiles are neither
// loaded nor computed, and every warp walks the same list of kept tiles.  A
// query tile with no kept key tile writes dQ = 0.
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
  static constexpr int QB_BYTES = NCH * BQ * 128;  // one prefetched Q or dO tile
  static constexpr int AVAIL = kMaxDynSmem - 512 - 1024 - 2 * QB_BYTES;
  static constexpr int STAGES = AVAIL / (2 * KV_BYTES) > 6 ? 6 : AVAIL / (2 * KV_BYTES);  // K_j + V_j each
  static constexpr int SMEM_BYTES = 1024 + 2 * QB_BYTES + STAGES * 2 * KV_BYTES;
  static constexpr int DQ_COL = 0, Q_COL = 128, DO_COL = 192, S_COL = 256, DP_COL = 320;  // dP: 3 x 64
  static constexpr int NDP = 3;  // dP buffers
  static constexpr int TMEM_COLS = 512;
  static constexpr int NUM_COMPUTE_WARPS = 8;
  static constexpr int NCT = 32 * NUM_COMPUTE_WARPS;
  static constexpr int PRODUCER_WARP = NUM_COMPUTE_WARPS;
  static constexpr int S_MMA_WARP = NUM_COMPUTE_WARPS + 1;
  static constexpr int DQ_MMA_WARP = NUM_COMPUTE_WARPS + 2;
  static constexpr int NUM_THREADS = 32 * (NUM_COMPUTE_WARPS + 3);
  // element pairs (of 16 per thread and key tile) whose exponentials use the
  // polynomial.  Without a block mask: the same in every row warp, one code
  // path for all of them, which measured faster than shares that differ per
  // sub-partition, and no share fastest (L = 8192: 0.49 ms against 0.51-0.52
  // for uniform 2 or 4 and 0.57-0.60 for 2-8 on the dQ / dP warp's
  // sub-partition only).  The block-mask instantiation keeps a dispatch per
  // sub-partition (POLY_MASKED on the dQ / dP warp's), which with no share
  // measured fastest there (random half of the blocks: backward 0.66 ms,
  // against 0.69 with 8 pairs and 0.73 with the single call), and gives the
  // same arithmetic as the unmasked kernel: an all-ones mask reproduces the
  // unmasked results bit for bit.
#ifndef GBATTN_DQ_POLY
  static constexpr int POLY = 0;
#else
  static constexpr int POLY = GBATTN_DQ_POLY;
#endif
#ifndef GBATTN_DQ_POLY_MASKED
  static constexpr int POLY_MASKED = 0;
#else
  static constexpr int POLY_MASKED = GBATTN_DQ_POLY_MASKED;
#endif
  static_assert(POLY >= 0 && POLY <= 16 && POLY_MASKED >= 0 && POLY_MASKED <= 16, "polynomial share");
  static_assert(D <= 128, "dQ, Q, dO and the S / dP buffers fill TMEM at D = 128");
  static_assert(STAGES >= NDP + 1, "dP of tile j+3 is issued while K_j is still in use");
};

// Work item w of the list (heaviest query tiles first): query tile and
// (batch, head) index.
struct Dq3Item {
  int qt, bh;
};
__device__ __forceinline__ Dq3Item dq3_item(int w, int BH, int n_qtiles) {
  const int t = w / BH;
  return {n_qtiles - 1 - t, w - t * BH};
}
constexpr int kDq3ItemRing = 4;  // rounds whose item index a CTA keeps in shared memory

template <int D, bool BF16, bool CAUSAL, bool MASKED>
__global__ void __launch_bounds__(Dq3Geom<D>::NUM_THREADS, 1)
    attn_bwd_dq3_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmdO,
                        const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                        const __grid_constant__ CUtensorMap tmdQ, const BwdParams p) {
  using Gm = Dq3Geom<D>;
  using E = Elem<BF16>;
  constexpr int BQ = Gm::BQ, BK = Gm::BK, NCH = Gm::NCH, ST = Gm::STAGES, NDP = Gm::NDP;

  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t bar_qbfull, bar_qbfree, bar_qread, bar_qready, bar_kvfull[ST], bar_kvempty[ST], bar_sfull, bar_sfree,
      bar_dpfull[NDP], bar_dsready[NDP], bar_dqdone, bar_mfin[2];
  __shared__ uint64_t bar_item[kDq3ItemRing];
  __shared__ volatile int item_ring[kDq3ItemRing];  // work item of round r in slot r % 4 (-1: no more)
  __shared__ uint32_t tmem_slot;
  __shared__ volatile int abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t sQb = sbase;                // prefetched Q tile; an item's dQ on its way out
  const uint32_t sDOb = sQb + Gm::QB_BYTES;  // prefetched dO tile
  const uint32_t sK0 = sDOb + Gm::QB_BYTES;  // stage s: K at sK0 + 2s * KV_BYTES, V right after

  const int BH = p.B * p.Hq;
  const int n_items = p.n_qtiles * BH;
  // key tiles of query tile qt
  auto n_kv_of = [&](int qt) {
    const int q_hi = min(qt * BQ + BQ, p.Lq);
    const int kv_end = CAUSAL ? min(p.Lk, q_hi + p.off) : p.Lk;
    return (kv_end + BK - 1) / BK;
  };
  static_assert(BQ == kMaskBlock && 2 * BK == kMaskBlock, "query tile = mask block, key tile = half a block");
  // key tile j of query tile qt is computed (block mask)
  auto keep = [&](int qt, int j) { return !MASKED || mask_keep(p, qt, j >> 1); };
  // number of computed key tiles of query tile qt (warp-collective)
  auto n_kept = [&](int qt) { return count_kept<MASKED>([&](int j) { return keep(qt, j); }, 0, n_kv_of(qt)); };
  const WaitGuard g{&abort_flag, p.status, p.limit_ns};
  // the work item of round r, as the producer published it; -1 ends the
  // CTA's loop (also once a wait has run out, so no loop outlives an abort)
  auto round_item = [&](int r) {
    mbar_wait(smem_u32(&bar_item[r % kDq3ItemRing]), (r / kDq3ItemRing) & 1, g, wait_code<76>());
    return abort_flag ? -1 : item_ring[r % kDq3ItemRing];
  };
  // extents for the debug build's index checks: rows of q / dq / lse /
  // delta, of dk / dv, and of the k / v buffers (pitch kv_pitch per head)
  [[maybe_unused]] const size_t n_qrows = static_cast<size_t>(p.B) * p.Hq * p.Lq;
  [[maybe_unused]] const size_t n_krows = static_cast<size_t>(p.B) * p.Hkv * p.Lk;
  [[maybe_unused]] const size_t n_kvbuf = (static_cast<size_t>(p.B) * p.Hkv - 1) * p.kv_pitch + p.Lk;

  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(smem_u32(&bar_qbfull), 1);
    mbar_init(smem_u32(&bar_qbfree), Gm::NCT);
    mbar_init(smem_u32(&bar_qread), Gm::NCT);  // every row thread has read the Q / dO buffer
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
    for (int i = 0; i < 2; ++i) mbar_init(smem_u32(&bar_mfin[i]), 1);
    for (int i = 0; i < kDq3ItemRing; ++i) mbar_init(smem_u32(&bar_item[i]), 1);
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
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmdO);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      tma_prefetch_desc(&tmdQ);
    }
    __syncwarp();
    int nqb = 0;  // Q / dO prefetches issued
    // dQ of item d, which the row threads staged in the Q prefetch buffer
    // (32-row tiles in the map's swizzled layout: 64-column chunk h of rows
    // 32 * qd .. +31 at sQb + h * BQ * 128 + qd * 32 * 128), written out with
    // one TMA store per tile; the buffer may take the next Q once they have
    // read it.  Rows past Lq are outside the map and are not written.
    auto store_dq = [&](const Dq3Item& d) {
      if (lane == 0) {
        for (int h = 0; h < NCH; ++h)
          for (int qd = 0; qd < 4; ++qd)
            if (d.qt * BQ + qd * 32 < p.Lq)
              tma_store_3d(&tmdQ, sQb + h * (BQ * 128) + qd * (32 * 128), h * 64, d.qt * BQ + qd * 32, d.bh);
        bulk_commit_group();
        bulk_wait_read_all();
      }
      __syncwarp();
    };
    auto load_q = [&](int w) {
      const Dq3Item it = dq3_item(w, BH, p.n_qtiles);
      ++nqb;
      mbar_arrive_expect_tx_w(smem_u32(&bar_qbfull), 2 * Gm::QB_BYTES);
      for (int c = 0; c < NCH; ++c) {
        tma_load_3d_w(sQb + c * BQ * 128, &tmQ, smem_u32(&bar_qbfull), c * 64, it.qt * BQ, it.bh);
        tma_load_3d_w(sDOb + c * BQ * 128, &tmdO, smem_u32(&bar_qbfull), c * 64, it.qt * BQ, it.bh);
      }
    };
    // the next item from the global counter (warp-collective), -1 past the end
    auto take_item = [&]() {
      int t = 0;
      if (lane == 0) t = atomicAdd(p.sched, 1);
      t = __shfl_sync(0xffffffffu, t, 0);
      return t < n_items ? t : -1;
    };
    auto publish = [&](int r, int w) {
      if (lane == 0) {
        item_ring[r % kDq3ItemRing] = w;
        mbar_arrive(smem_u32(&bar_item[r % kDq3ItemRing]));
      }
      __syncwarp();
    };
    RingPos<ST> kv;  // stage of the next key tile
    bool wrapped = false;  // the ring has been filled once: stages must be freed first
    int r = 0;
    Dq3Item prev{};  // the item of the previous round
    int w = take_item();
    publish(0, w);
    if (w >= 0) load_q(w);
    for (; w >= 0 && !abort_flag; ++r) {
      const Dq3Item it = dq3_item(w, BH, p.n_qtiles);
      const int b = it.bh / p.Hq, hq = it.bh - b * p.Hq;
      const int zkv = b * p.Hkv + hq / p.G;
      const int n_kv = n_kv_of(it.qt);
      auto kw = kept_walk<MASKED>([&](int j) { return keep(it.qt, j); }, n_kv);
      for (int j = kw.first(0); j < n_kv; j = kw.next(j)) {
        const int s = kv.slot;
        if (kv.slot == 0 && kv.phase == 1) wrapped = true;
        if (wrapped) mbar_wait(smem_u32(&bar_kvempty[s]), kv.phase ^ 1u, g, wait_code<61>());
        __syncwarp();
        if (abort_flag) break;  // after an abort no further copy is issued
        const uint32_t bar = smem_u32(&bar_kvfull[s]);
        const uint32_t dK = sK0 + 2 * s * Gm::KV_BYTES;
        mbar_arrive_expect_tx_w(bar, 2 * Gm::KV_BYTES);
        for (int c = 0; c < NCH; ++c) {
          tma_load_3d_w(dK + c * BK * 128, &tmK, bar, c * 64, j * BK, zkv);
          tma_load_3d_w(dK + Gm::KV_BYTES + c * BK * 128, &tmV, bar, c * 64, j * BK, zkv);
        }
        kv.next();
      }
      // The row threads copied this item's Q / dO out of the buffer when the
      // item started (after every MMA of round r - 1 had completed, so every
      // warp has read round r - 1's slot) and staged round r - 1's dQ in it:
      // round r + 1 may take the slot of round r - 3, and once that dQ is
      // out, the buffer the next item's Q / dO.
      w = take_item();
      mbar_wait(smem_u32(&bar_qbfree), r & 1, g, wait_code<72>());
      __syncwarp();
      if (r > 0 && !abort_flag) store_dq(prev);
      prev = it;
      publish(r + 1, w);
      if (w >= 0 && !abort_flag) load_q(w);
    }
    // the last item's dQ, staged after its last MMA
    if (r > 0 && !abort_flag) {
      mbar_wait(smem_u32(&bar_qbfree), r & 1, g, wait_code<74>());
      __syncwarp();
      if (!abort_flag) store_dq(prev);
    }
    if (lane == 0) bulk_wait_all();
    __syncwarp();
    // the last Q / dO prefetch and the last ST issued stages (fewer if the
    // ring never wrapped; a stage is refilled only after its release, so each
    // holds at most one copy in flight)
    if (nqb > 0) mbar_wait_drain(smem_u32(&bar_qbfull), (nqb - 1) & 1);
    for (int u = 0; u < ST; ++u) {
      kv.slot = kv.slot == 0 ? ST - 1 : kv.slot - 1;
      if (kv.slot == ST - 1) {
        if (!wrapped && kv.phase == 0) break;  // before the first stage issued
        kv.phase ^= 1u;
      }
      mbar_wait_drain(smem_u32(&bar_kvfull[kv.slot]), kv.phase);
    }
    __syncwarp();
  } else if (warp == Gm::S_MMA_WARP) {
    // ---------------- S = Q K^T issuer (A operand Q from tensor memory) ----------------
    constexpr uint32_t IDESC_S = make_idesc_f16(128, BK, BF16, false, false);
    const uint64_t dKk = make_sdesc_sw128(sK0, 16, 1024);  // K stage 0, K-major
    RingPos<ST> kv;       // stage of the next key tile
    uint32_t sphase = 0;  // parity of the S buffer's next use
    bool first = true;
    for (int r = 0, w = round_item(0); w >= 0; w = round_item(++r)) {
      const int nk = n_kept(dq3_item(w, BH, p.n_qtiles).qt);
      // this item's Q is in tensor memory
      mbar_wait(smem_u32(&bar_qready), r & 1, g, wait_code<63>());
      for (int j = 0; j < nk; ++j, kv.next()) {
        const int s = kv.slot;
        // every row thread has loaded the previous S from the buffer
        if (!first) mbar_wait(smem_u32(&bar_sfree), sphase ^ 1u, g, wait_code<64>());
        first = false;
        sphase ^= 1u;
        mbar_wait(smem_u32(&bar_kvfull[s]), kv.phase, g, wait_code<65>());
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
    }
    // every MMA this warp issued is complete before tensor memory is released
    mma_commit_w(smem_u32(&bar_mfin[0]));
    mbar_wait_drain(smem_u32(&bar_mfin[0]), 0);
    __syncwarp();
  } else if (warp == Gm::DQ_MMA_WARP) {
    // ---------------- dQ += dS K and dP = dO V^T issuer ----------------
    constexpr uint32_t IDESC_S = make_idesc_f16(128, BK, BF16, false, false);
    constexpr uint32_t IDESC_DQ = make_idesc_f16(128, D, BF16, false, true);
    const uint64_t dVk = make_sdesc_sw128(sK0 + Gm::KV_BYTES, 16, 1024);  // V stage 0, K-major
    const uint64_t dKm = make_sdesc_sw128(sK0, BK * 128, 1024);           // K stage 0, MN-major
    RingPos<ST> kv, kv_dp;  // stages of the next dQ and the next dP key tile
    RingPos<NDP> db, db_dp;  // dP buffers of the next dQ and the next dP
    // dP of the next key tile to load into its dP buffer
    auto issue_dp = [&]() {
      const int s = kv_dp.slot, buf = db_dp.slot;
      mbar_wait(smem_u32(&bar_kvfull[s]), kv_dp.phase, g, wait_code<67>());
      __syncwarp();
      tc_fence_after_sync();
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t vo = 2 * s * Gm::KV_BYTES + (kk >> 2) * (BK * 128) + (kk & 3) * 32;
        mma_ts_w(tmem + Gm::DP_COL + buf * BK, tmem + Gm::DO_COL + kk * 8, sdesc_add(dVk, vo), IDESC_S,
                 kk > 0 ? 1u : 0u);
      }
      mma_commit_w(smem_u32(&bar_dpfull[buf]));
      kv_dp.next();
      db_dp.next();
    };
    for (int r = 0, w = round_item(0); w >= 0; w = round_item(++r)) {
      const int nk = n_kept(dq3_item(w, BH, p.n_qtiles).qt);
      // this item's dO is in tensor memory
      mbar_wait(smem_u32(&bar_qready), r & 1, g, wait_code<66>());
      for (int j = 0; j < NDP && j < nk; ++j) issue_dp();
      for (int j = 0; j < nk; ++j, kv.next(), db.next()) {
        const int s = kv.slot, buf = db.slot;
        mbar_wait(smem_u32(&bar_dsready[buf]), db.phase, g, wait_code<68>());
        __syncwarp();
        tc_fence_after_sync();
        // A operand: 16 keys per K step; keys 32h..32h+31 of warpgroup h sit as
        // pairs in columns 32h..32h+15 of the dP buffer.
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk) {
          const uint32_t acol = Gm::DP_COL + buf * BK + (kk >> 1) * 32 + (kk & 1) * 8;
          mma_ts_w(tmem + Gm::DQ_COL, tmem + acol, sdesc_add(dKm, 2 * s * Gm::KV_BYTES + kk * 2048), IDESC_DQ,
                   (j > 0 || kk > 0) ? 1u : 0u);
        }
        // this warp's dP(t) and dQ(t) are its last reads of the stage
        mma_commit_w(smem_u32(&bar_kvempty[s]));
        // dP three tiles ahead overwrites the buffer behind dQ, which reads its dS
        if (j + NDP < nk) issue_dp();
      }
      // Every S MMA of the item completed before its last dS was ready, so
      // this commit covers all of the item's MMAs.
      mma_commit_w(smem_u32(&bar_dqdone));
    }
    mma_commit_w(smem_u32(&bar_mfin[1]));
    mbar_wait_drain(smem_u32(&bar_mfin[1]), 0);
    __syncwarp();
  } else {
    // ---------------- row threads ----------------
    const int quad = warp & 3;   // TMEM lane quadrant (query rows)
    const int half = warp >> 2;  // key columns 32*half .. +31 of each tile
    const int rr_ = quad * 32 + lane;  // row of the query tile
    const uint32_t lrow = static_cast<uint32_t>(quad * 32) << 16;
    const float sl2 = p.scale_log2;
    const uint64_t sl2x2 = f2_pack(sl2, sl2);
    constexpr int HALF = D / 2;  // elements of a Q / dO row this thread copies
    uint32_t sphase = 0;  // parity of the S buffer's next fill
    RingPos<NDP> db;      // dP buffer of the next key tile
    // Q and dO rows of the item of round rn from the prefetch buffer (TMA
    // layout: 64-column chunks of 128-byte rows, 16-byte units swizzled by
    // row % 8; zeros past Lq and past D) into tensor memory: this warp copies
    // elements [half*D/2, (half+1)*D/2) of its 32 rows as 16-bit pairs.  No
    // MMA of the previous item reads them any more (its final commit has
    // completed).  The first item hands the buffer back at once; later ones
    // after the epilogue has staged the previous item's dQ in it.
    auto copy_q = [&](int rn, bool release) {
      mbar_wait(smem_u32(&bar_qbfull), rn & 1, g, wait_code<73>());
      uint32_t qa[HALF / 2], oa[HALF / 2];
#pragma unroll
      for (int v = 0; v < HALF / 8; ++v) {
        const int e = half * HALF + 8 * v;  // first element of this 16-byte unit
        const uint32_t off = (e / 64) * (BQ * 128) + rr_ * 128 + ((((e % 64) / 8) ^ (rr_ & 7)) * 16);
        const uint4 x = ld_shared_v4(sQb + off), y = ld_shared_v4(sDOb + off);
        qa[4 * v + 0] = x.x, qa[4 * v + 1] = x.y, qa[4 * v + 2] = x.z, qa[4 * v + 3] = x.w;
        oa[4 * v + 0] = y.x, oa[4 * v + 1] = y.y, oa[4 * v + 2] = y.z, oa[4 * v + 3] = y.w;
      }
      // the producer may refill the buffer once every row thread has read it
      if (release) {
        fence_proxy_async_smem();
        mbar_arrive(smem_u32(&bar_qbfree));
      }
      // HALF / 2 packed columns: 16, 24 or 32 (D = 64, 96, 128)
#pragma unroll
      for (int c = 0; c + 16 <= HALF / 2; c += 16) {
        uint32_t t16[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) t16[i] = qa[c + i];
        tmem_st16(tmem + lrow + Gm::Q_COL + half * (HALF / 2) + c, t16);
#pragma unroll
        for (int i = 0; i < 16; ++i) t16[i] = oa[c + i];
        tmem_st16(tmem + lrow + Gm::DO_COL + half * (HALF / 2) + c, t16);
      }
      if constexpr ((HALF / 2) % 16 == 8) {
        constexpr int c = HALF / 2 - 8;
        uint32_t t8[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) t8[i] = qa[c + i];
        tmem_st8(tmem + lrow + Gm::Q_COL + half * (HALF / 2) + c, t8);
#pragma unroll
        for (int i = 0; i < 8; ++i) t8[i] = oa[c + i];
        tmem_st8(tmem + lrow + Gm::DO_COL + half * (HALF / 2) + c, t8);
      }
      tmem_st_wait();
      tc_fence_before_sync();
      mbar_arrive(smem_u32(&bar_qready));
    };
    if (round_item(0) >= 0) copy_q(0, true);
    for (int r = 0, w = round_item(0); w >= 0; w = round_item(++r)) {
      const Dq3Item it = dq3_item(w, BH, p.n_qtiles);
      const int q0 = it.qt * BQ;
      const int qi = q0 + rr_;
      const int n_kv = n_kv_of(it.qt);
      const int nk = n_kept(it.qt);
      const size_t row = static_cast<size_t>(it.bh) * p.Lq + qi;
      const float lse_r = qi < p.Lq && dbg_in_range(row, 1, n_qrows, p.status, 7) ? p.lse[row] : 0.f;
      const float dlt_r = qi < p.Lq && dbg_in_range(row, 1, n_qrows, p.status, 8) ? p.delta[row] : 0.f;
      const uint64_t nlse2 = f2_pack(-lse_r, -lse_r), dlt2 = f2_pack(dlt_r, dlt_r);
      const int lim = CAUSAL ? min(qi + p.off, p.Lk - 1) : p.Lk - 1;
      auto kw = kept_walk<MASKED>([&](int j) { return keep(it.qt, j); }, n_kv);
      for (int j = kw.first(0); j < n_kv; j = kw.next(j)) {
        const int buf = db.slot;
        const uint32_t dph = db.phase;
        db.next();
        mbar_wait(smem_u32(&bar_sfull), sphase, g, wait_code<69>());
        sphase ^= 1u;
        mbar_wait(smem_u32(&bar_dpfull[buf]), dph, g, wait_code<71>());
        __syncwarp();
        tc_fence_after_sync();
        const int kc0 = j * BK + half * 32;  // first key of this thread's columns
        const bool need_mask = (CAUSAL && (j * BK + BK - 1 > q0 + p.off)) || (j * BK + BK > p.Lk);
        const uint32_t dcol = tmem + lrow + Gm::DP_COL + buf * BK + half * 32;
        uint32_t sr[32], dr[32];
        tmem_ld32(tmem + lrow + Gm::S_COL + half * 32, sr);
        tmem_ld32(dcol, dr);
        tmem_ld_wait(sr);
        reg_fence(dr);
        // S(t) is in registers: the S warp may overwrite the buffer
        tc_fence_before_sync();
        mbar_arrive(smem_u32(&bar_sfree));
        uint32_t pk[16];
        // NPOLY of the 16 pairs, spread evenly, use the polynomial
        auto ds_tile = [&](auto npoly_tag) {
          constexpr int NPOLY = decltype(npoly_tag)::value;
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            float x0, x1, p0, p1;
            f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[2 * i]), __uint_as_float(sr[2 * i + 1])), sl2x2, nlse2), x0,
                      x1);
            if ((i + 1) * NPOLY / 16 > i * NPOLY / 16) {
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
        if constexpr (MASKED) {
          if (quad == 1)  // sub-partition of the S warp
            ds_tile(std::integral_constant<int, 0>{});
          else if (quad == 2)  // sub-partition of the dQ / dP warp
            ds_tile(std::integral_constant<int, Gm::POLY_MASKED>{});
          else
            ds_tile(std::integral_constant<int, 0>{});
        } else {
          ds_tile(std::integral_constant<int, Gm::POLY>{});
        }
        tmem_st16(dcol, pk);
        tmem_st_wait();
        tc_fence_before_sync();
        mbar_arrive(smem_u32(&bar_dsready[buf]));
      }
      // epilogue of the item: every MMA of the item is complete
      mbar_wait(smem_u32(&bar_dqdone), r & 1, g, wait_code<70>());
      __syncwarp();
      tc_fence_after_sync();
      // the next item's Q and dO first, so that its first S and dP products
      // run while this item's dQ is read out and stored (copying them right
      // after the item's last dS instead measured 32% slower at D = 96 and no
      // faster at D = 128)
      if (round_item(r + 1) >= 0) copy_q(r + 1, false);
      // Every row thread has read the prefetch buffer: it now stages this
      // item's dQ, warp (quad, half) writing 64-column chunk `half` of its 32
      // rows, for the producer's TMA stores.  Staging through shared memory
      // keeps the stores off the load/store unit (a store per row from every
      // thread touches 32 rows' lines per instruction).
      mbar_arrive(smem_u32(&bar_qread));
      mbar_wait(smem_u32(&bar_qread), r & 1, g, wait_code<75>());
      if (half < NCH) {
        const uint32_t stg = sQb + half * (BQ * 128) + quad * (32 * 128) + lane * 128;
#pragma unroll 1
        for (int c = 2 * half; c < 2 * half + 2 && c < D / 32; ++c) {
          uint32_t rr[32];
          if (nk > 0) {  // same for the whole CTA: tcgen05.ld is warp-collective
            tmem_ld32(tmem + lrow + Gm::DQ_COL + c * 32, rr);
            tmem_ld_wait(rr);
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) rr[i] = 0u;  // no kept key tile: dQ = 0
          }
          uint32_t pk[16];
          pack_row32<BF16>(rr, p.scale, pk);
          stage_row16_sw128(stg, lane, (c & 1) * 4, pk);
        }
      }
      fence_proxy_async_smem();
      mbar_arrive(smem_u32(&bar_qbfree));
      // The next item's first dQ MMA overwrites these columns; it is issued
      // after this thread's next dS arrival, which follows these loads.
      tc_fence_before_sync();
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == Gm::S_MMA_WARP) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, Gm::TMEM_COLS);
  }
  if (threadIdx.x == 0) {
    // Launched behind the dK/dV kernel, this grid may not finish before it.
    grid_dependency_wait();
    // The last CTA to finish puts the work counter back to zero: every CTA
    // has taken its last item by now.
    __threadfence();
    if (atomicAdd(p.sched + 1, 1) == static_cast<int>(gridDim.x) - 1) {
      p.sched[0] = 0;
      p.sched[1] = 0;
      __threadfence();
    }
  }
}

}  // namespace gbattn
