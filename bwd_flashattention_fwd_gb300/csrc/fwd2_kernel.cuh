// Forward attention with saved base-2 log-sum-exp, two query tiles per CTA
// (head dims up to 128).
//
// Same mathematics as fwd_kernel.cuh (online softmax over key tiles in the
// log2 domain: "When the Bottleneck Moved", section 3; "feat(attention):
// complete Flash Attention VJP implementation", section "Background"), laid
// out so the tensor cores and the softmax work overlap:
//   * the CTA owns 256 query rows as two 128-row tiles that share every K/V
//     tile, with one softmax warpgroup per tile;
//   * keys come in tiles of BK = 64 and each query tile has two S buffers in
//     tensor memory, so S_t for key tile j+1 (and j+2) is computed while the
//     softmax warpgroup works on tile j;  O_0, O_1 (fp32, 128 columns each)
//     and S_0[2], S_1[2] (fp32, 64 columns each) fill the 512 TMEM columns;
//   * P_t (16-bit pairs) is written back over the first 32 columns of its S
//     buffer, which the warpgroup has already read; the MMA that next writes
//     that buffer is issued after O_t += P_t V_j by the same thread (tcgen05
//     MMAs of one CTA run in issue order);
//   * lazy rescaling: a row keeps its reference maximum m until a new tile
//     raises the row maximum by more than TAU = 8 (in log2 units), so P <= 2^8
//     and O / l are rescaled only on those (rare) tiles, after waiting for the
//     previous P V product.  The final O = acc / l and lse = m + log2 l use the
//     same reference, so the result is exact in exact arithmetic.
//
// Warp roles (352 threads): warps 0-3 softmax for tile 0, warps 4-7 for tile 1
// (thread = query row = TMEM lane), warp 8 TMA producer (Q once, then K_j and
// V_j together into one ring stage), warp 9 issues tile 0's MMAs and owns the
// TMEM allocation, warp 10 issues tile 1's MMAs.  Each MMA warp orders its
// own tile's S / P aliasing; splitting the issue over two warps halves the
// serial barrier-wait and commit overhead per key tile, which otherwise
// exceeds the tensor time of a 64-key step.
//
// The softmax works on packed pairs (.f32x2 fma / add) and takes the row
// maximum with three-input max, which keeps its instruction count, and so its
// share of the issue slots of the sub-partitions the MMA warps run on, low.
//
// Persistent: one CTA per SM walks a list of (256-row query pair, head) work
// items, heaviest first: each CTA starts with the item of its own index and
// takes the next from a global counter when its producer has issued the
// current one's copies, and hands the index to the other warps through a
// four-slot ring in shared memory (a static deal left the busiest CTA's
// key-tile loops ~8% above the median at L = 2048).  As soon as an item's last S MMAs have completed, the producer loads the next
// item's Q into the (then unused) Q buffer, and the MMA warps compute the next
// item's first S tiles while the softmax warps write out the current item's O
// and lse.  Barrier phases count key tiles and items over the CTA's life.
// O goes out through shared memory: each softmax warp converts its 32 rows
// into a 4 KB staging tile (64 columns at a time, in the swizzled layout of
// the output's tensor map) and one lane issues a TMA store, so the tensor
// pipe idles only briefly between items (a 16-byte store per row from every
// thread kept the load/store unit busy for ~3 us per item).  The staging
// costs one K/V ring stage, which measured free.
//
// MASKED: block-sparse variant ("feat(attention): complete Flash Attention
// VJP implementation", section "Sparse Block Masks"; the forward applies the
// same mask so that the saved lse matches the gradients).  Each 128-row query
// tile is one mask block and each key tile half of a 128-key block.  A key
// tile that both query tiles of the item mask is neither loaded nor computed;
// one that only one of them masks is computed and set to -inf for that tile.
// A row that sees no key gets O = 0 and lse = +inf.
#pragma once

#include "kernel_common.cuh"

namespace gbattn {

constexpr int kFwdItemRing = 4;  // rounds whose item index a CTA keeps in shared memory

template <int D>
struct Fwd2Geom {
  static constexpr int BQ = 128;  // rows per query tile; the CTA owns 2 tiles
  static constexpr int BK = 64;
  static constexpr int NCH = n_chunks(D);
  static constexpr int Q_BYTES = NCH * BQ * 128;
  static constexpr int KV_BYTES = NCH * BK * 128;
  // O staging: each softmax warp's 32 rows x 64 columns (16-bit), swizzled
  static constexpr int O_STG_BYTES = 32 * 128;
  static constexpr int AVAIL = kMaxDynSmem - 512 - 1024 - 2 * Q_BYTES - 8 * O_STG_BYTES;
  static constexpr int STAGES = AVAIL / (2 * KV_BYTES) > 6 ? 6 : AVAIL / (2 * KV_BYTES);  // K_j + V_j each
  static constexpr int SMEM_BYTES = 1024 + 2 * Q_BYTES + STAGES * 2 * KV_BYTES + 8 * O_STG_BYTES;
  static constexpr int TMEM_COLS = 512;
  static constexpr int NUM_THREADS = 352;
  static constexpr float TAU = 8.0f;
  __host__ __device__ static constexpr int o_col(int t) { return t * 128; }
  __host__ __device__ static constexpr int s_col(int t, int b) { return 256 + t * 128 + b * 64; }
  static_assert(D <= 128, "two O accumulators need D <= 128");
  // S for key tile j+2 is issued while K_j / V_j may still be in use
  static_assert(STAGES >= 3, "shared memory budget");
};

template <int D, bool BF16, bool CAUSAL, bool MASKED>
__global__ void __launch_bounds__(352, 1)
    attn_fwd2_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                     const FwdParams p) {
  using Gm = Fwd2Geom<D>;
  using E = Elem<BF16>;
  constexpr int BQ = Gm::BQ, BK = Gm::BK, NCH = Gm::NCH, ST = Gm::STAGES;

  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t bar_q, bar_qfree, bar_kvfull[ST], bar_kvempty[ST], bar_sfull[2][2], bar_pready[2][2],
      bar_odone[2], bar_done, bar_mfin[2];
  // work item of round r in slot r % 4 (-1: no more); bar_itemfree: every
  // consumer warp (the MMA and softmax warps) has read the slot
  __shared__ uint64_t bar_item[kFwdItemRing], bar_itemfree[kFwdItemRing];
  __shared__ volatile int item_ring[kFwdItemRing];
  __shared__ uint32_t tmem_slot;
  __shared__ volatile int abort_flag;

  // A kernel launched behind this one as a programmatic dependent (the delta
  // kernel) may take the SMs this grid frees; it waits for this grid to
  // complete before it reads anything.
  if (threadIdx.x == 0) grid_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t sQ = sbase;  // tile t at sQ + t * Q_BYTES
  const uint32_t sK0 = sQ + 2 * Gm::Q_BYTES;  // stage s: K at sK0 + 2s * KV_BYTES, V right after
  const uint32_t sO = sK0 + ST * 2 * Gm::KV_BYTES;  // softmax warp w's O staging at sO + w * O_STG_BYTES

  // work items: w -> (query pair pt, head bh), heaviest query pairs first;
  // n_qtiles counts 256-row pairs
  const int BH = p.B * p.Hq;
  const int n_items = p.n_qtiles * BH;
  auto item_pt = [&](int w) { return p.n_qtiles - 1 - w / BH; };
  auto item_bh = [&](int w) { return w - (w / BH) * BH; };
  auto n_kv_of = [&](int pt) {
    const int q_hi = min(pt * 2 * BQ + 2 * BQ, p.Lq);
    const int kv_end = CAUSAL ? min(p.Lk, q_hi + p.off) : p.Lk;
    return (kv_end + BK - 1) / BK;
  };
  static_assert(BQ == kMaskBlock && 2 * BK == kMaskBlock, "query tile = mask block, key tile = half a block");
  const int nqb = (p.Lq + kMaskBlock - 1) / kMaskBlock;
  // key tile j is visible to query tile t of pair pt as far as the block mask goes
  auto keep_t = [&](int pt, int t, int j) {
    return !MASKED || (2 * pt + t < nqb && mask_keep(p, 2 * pt + t, j >> 1));
  };
  // key tile j is computed for the pair (either query tile keeps it)
  auto keep = [&](int pt, int j) { return !MASKED || keep_t(pt, 0, j) || keep_t(pt, 1, j); };
  // computed key tiles of pair pt (warp-collective)
  auto n_kept = [&](int pt) { return count_kept<MASKED>([&](int j) { return keep(pt, j); }, 0, n_kv_of(pt)); };
  const WaitGuard g{&abort_flag, p.status, p.limit_ns};
  // The work item of round r, as the producer published it (warp-collective);
  // -1 ends the loop (also once a wait has run out, so no loop outlives an
  // abort).  The warp hands the slot back once every lane has read it.
  auto round_item = [&](int r) {
    const int slot = r % kFwdItemRing;
    mbar_wait(smem_u32(&bar_item[slot]), (r / kFwdItemRing) & 1, g, wait_code<36>());
    const int w = abort_flag ? -1 : item_ring[slot];
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&bar_itemfree[slot]));
    return w;
  };
  // extents for the debug build's index checks: rows of q / o / lse
  [[maybe_unused]] const size_t n_qrows = static_cast<size_t>(p.B) * p.Hq * p.Lq;

  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(smem_u32(&bar_q), 1);
    mbar_init(smem_u32(&bar_qfree), 2);  // one commit per MMA warp after its item's last S
    // A stage (K_j, V_j) is free once both tiles' MMAs that read it
    // completed: one commit from each MMA warp, after its P_t V_j.
    for (int s = 0; s < ST; ++s) {
      mbar_init(smem_u32(&bar_kvfull[s]), 1);
      mbar_init(smem_u32(&bar_kvempty[s]), 2);
    }
    for (int t = 0; t < 2; ++t) {
      for (int bb = 0; bb < 2; ++bb) {
        mbar_init(smem_u32(&bar_sfull[t][bb]), 1);
        mbar_init(smem_u32(&bar_pready[t][bb]), 128);
      }
      mbar_init(smem_u32(&bar_odone[t]), 1);
    }
    mbar_init(smem_u32(&bar_done), 2);
    for (int t = 0; t < 2; ++t) mbar_init(smem_u32(&bar_mfin[t]), 1);
    for (int i = 0; i < kFwdItemRing; ++i) {
      mbar_init(smem_u32(&bar_item[i]), 1);
      mbar_init(smem_u32(&bar_itemfree[i]), 10);  // warps 0-7 and 9-10
    }
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc(smem_u32(&tmem_slot), Gm::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = tmem_slot;

  if (warp == 8) {
    // ---------------- TMA producer (whole warp, one elected lane issues) ----------------
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      tma_prefetch_desc(&tmO);
    }
    __syncwarp();
    RingPos<ST> st;  // stage of the next key tile
    int issued = 0;  // key tiles issued (all items)
    int nq = 0;      // items whose Q was loaded
    // The next item from the global counter (warp-collective), -1 past the
    // end; each CTA's first item is its own index (the grid has at most one
    // CTA per item), so the counter starts behind them.
    auto take_item = [&]() {
      int t = 0;
      if (lane == 0) t = atomicAdd(p.sched, 1);
      t = __shfl_sync(0xffffffffu, t, 0) + static_cast<int>(gridDim.x);
      return t < n_items ? t : -1;
    };
    // round r's item into its ring slot, once every consumer warp has read
    // the round that used the slot before
    auto publish = [&](int r, int w) {
      const int slot = r % kFwdItemRing;
      if (r >= kFwdItemRing)
        mbar_wait(smem_u32(&bar_itemfree[slot]), ((r / kFwdItemRing) - 1) & 1, g, wait_code<95>());
      __syncwarp();
      if (lane == 0) {
        item_ring[slot] = abort_flag ? -1 : w;
        mbar_arrive(smem_u32(&bar_item[slot]));
      }
      __syncwarp();
    };
    int w = static_cast<int>(blockIdx.x);
    publish(0, w);
    // After an abort (a wait ran out) no further copy is issued, so the
    // drains below cover every copy still in flight.
    for (int r = 0; w >= 0 && !abort_flag; ++r) {
      const int pt = item_pt(w), bh = item_bh(w);
      const int b = bh / p.Hq, hq = bh - b * p.Hq;
      const int zkv = b * p.Hkv + hq / p.G;
      const int q0 = pt * 2 * BQ;
      const int n_kv = n_kv_of(pt);
      // the previous item's S MMAs, the only readers of Q, are complete
      if (r > 0) mbar_wait(smem_u32(&bar_qfree), (r - 1) & 1, g, wait_code<30>());
      __syncwarp();
      if (abort_flag) break;
      ++nq;
      mbar_arrive_expect_tx_w(smem_u32(&bar_q), 2 * Gm::Q_BYTES);
      for (int t = 0; t < 2; ++t)
        for (int c = 0; c < NCH; ++c)
          tma_load_3d_w(sQ + t * Gm::Q_BYTES + c * BQ * 128, &tmQ, smem_u32(&bar_q), c * 64, q0 + t * BQ, bh);
      auto kw = kept_walk<MASKED>([&](int j) { return keep(pt, j); }, n_kv);
      for (int j = kw.first(0); j < n_kv; j = kw.next(j)) {
        const int s = st.slot;
        if (issued >= ST) mbar_wait(smem_u32(&bar_kvempty[s]), st.phase ^ 1u, g, wait_code<31>());
        __syncwarp();
        if (abort_flag) break;
        const uint32_t bar = smem_u32(&bar_kvfull[s]);
        const uint32_t dK = sK0 + 2 * s * Gm::KV_BYTES;
        mbar_arrive_expect_tx_w(bar, 2 * Gm::KV_BYTES);
        for (int c = 0; c < NCH; ++c) {
          tma_load_3d_w(dK + c * BK * 128, &tmK, bar, c * 64, j * BK, zkv);
          tma_load_3d_w(dK + Gm::KV_BYTES + c * BK * 128, &tmV, bar, c * 64, j * BK, zkv);
        }
        st.next();
        ++issued;
      }
      // the next item, published while the MMA warps still work on this one
      w = take_item();
      publish(r + 1, w);
    }
    // the last ST issued stages (each slot holds at most one copy in
    // flight: a stage is refilled only after its release), and the last Q
    for (int u = 0; u < ST && u < issued; ++u) {
      if (st.slot == 0) st.phase ^= 1u;
      st.slot = (st.slot == 0 ? ST : st.slot) - 1;
      mbar_wait_drain(smem_u32(&bar_kvfull[st.slot]), st.phase);
    }
    if (nq > 0) mbar_wait_drain(smem_u32(&bar_q), (nq - 1) & 1);
    __syncwarp();
  } else if (warp == 9 || warp == 10) {
    // ---------------- MMA issuers: warp 9 for tile 0, warp 10 for tile 1 ----------------
    const int t = warp - 9;
    constexpr uint32_t IDESC_QK = make_idesc_f16(128, BK, BF16, false, false);
    constexpr uint32_t IDESC_PV = make_idesc_f16(128, D, BF16, false, true);
    const uint64_t dQd = make_sdesc_sw128(sQ + t * Gm::Q_BYTES, 16, 1024);  // this tile's Q, K-major
    const uint64_t dKk = make_sdesc_sw128(sK0, 16, 1024);                         // K stage 0, K-major
    const uint64_t dVm = make_sdesc_sw128(sK0 + Gm::KV_BYTES, BK * 128, 1024);    // V stage 0, MN-major
    RingPos<ST> st_s, st_pv;  // stages of the next S_t and of the next P_t V
    int ts = 0, tp = 0;       // key tiles (all items) of the next S_t and of the next P_t V
    // S_t of the next key tile; the wait on the stage also covers V_j for P_t V_j
    auto issue_s = [&]() {
      const int s = st_s.slot, bb = ts & 1;
      mbar_wait(smem_u32(&bar_kvfull[s]), st_s.phase, g, wait_code<34>());
      st_s.next();
      ++ts;
      __syncwarp();
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t qo = (kk >> 2) * (BQ * 128) + (kk & 3) * 32;
        const uint32_t ko = 2 * s * Gm::KV_BYTES + (kk >> 2) * (BK * 128) + (kk & 3) * 32;
        mma_ss_w(tmem + Gm::s_col(t, bb), sdesc_add(dQd, qo), sdesc_add(dKk, ko), IDESC_QK, kk > 0 ? 1u : 0u);
      }
      mma_commit_w(smem_u32(&bar_sfull[t][bb]));
    };
    // P_t V_j of key tile j of an item with n_kv key tiles
    auto issue_pv = [&](int j, int n_kv) {
      const int s = st_pv.slot, bb = tp & 1;
      const uint32_t ph = (tp >> 1) & 1;
      st_pv.next();
      ++tp;
      mbar_wait(smem_u32(&bar_pready[t][bb]), ph, g, wait_code<35>());
      __syncwarp();
      tc_fence_after_sync();
#pragma unroll
      for (int kk = 0; kk < BK / 16; ++kk)
        mma_ts_w(tmem + Gm::o_col(t), tmem + Gm::s_col(t, bb) + kk * 8,
                 sdesc_add(dVm, 2 * s * Gm::KV_BYTES + kk * 2048), IDESC_PV, (j > 0 || kk > 0) ? 1u : 0u);
      // this thread's S_t(j) and P_t V_j are the last reads of the stage
      mma_commit_w(smem_u32(&bar_kvempty[s]));
      // A rescale on the last key tile needs this product done; earlier
      // rescales use the next tile's S barrier, which covers it.
      if (j == n_kv - 2) mma_commit_w(smem_u32(&bar_odone[t]));
    };
    int r = 0;
    for (int w = round_item(0); w >= 0; w = round_item(++r)) {
      const int n_kv = n_kept(item_pt(w));  // computed key tiles of the item
      // this item's Q is in shared memory
      mbar_wait(smem_u32(&bar_q), r & 1, g, wait_code<33>());
      __syncwarp();
      tc_fence_after_sync();
      for (int j = 0; j < 2 && j < n_kv; ++j) {
        issue_s();
        if (j == n_kv - 1) mma_commit_w(smem_u32(&bar_qfree));  // last read of this item's Q
      }
      for (int j = 0; j < n_kv; ++j) {
        issue_pv(j, n_kv);
        if (j + 2 < n_kv) {
          issue_s();
          if (j + 2 == n_kv - 1) mma_commit_w(smem_u32(&bar_qfree));
        }
      }
      if (n_kv == 0) mma_commit_w(smem_u32(&bar_qfree));  // nothing reads this item's Q
      mma_commit_w(smem_u32(&bar_done));
    }
    // every MMA this warp issued is complete before tensor memory is released
    mma_commit_w(smem_u32(&bar_mfin[t]));
    mbar_wait_drain(smem_u32(&bar_mfin[t]), 0);
    __syncwarp();
  } else {
    // ---------------- softmax warpgroups ----------------
    const int t = warp >> 2;  // query tile
    const int quad = warp & 3;
    const int rt = quad * 32 + lane;  // row of the query tile
    const uint32_t lrow = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t o_col = tmem + lrow + Gm::o_col(t);
    const float sl2 = p.scale_log2;
    int ts = 0;             // key tiles (all items) seen so far
    uint32_t odone_ph = 0;  // parity of the next item-end product barrier
    int r = 0;
    for (int w = round_item(0); w >= 0; w = round_item(++r)) {
      const int bh = item_bh(w);
      const int q0t = item_pt(w) * 2 * BQ + t * BQ;
      const int qi = q0t + rt;
      const int pt = item_pt(w);
      const int n_kv = n_kv_of(pt);
      const int nk = n_kept(pt);
      const int lim = CAUSAL ? min(qi + p.off, p.Lk - 1) : p.Lk - 1;  // last visible key
      float m = -INFINITY, l = 0.f;
      auto kw = kept_walk<MASKED>([&](int j) { return keep(pt, j); }, n_kv);
      for (int j = kw.first(0), kc = 0; j < n_kv; j = kw.next(j), ++kc) {
        const int k = MASKED ? kc : j;  // computed key tiles before this one
        const int T = ts + k;
        const int bb = T & 1;
        const uint32_t s_col = tmem + lrow + Gm::s_col(t, bb);
        mbar_wait(smem_u32(&bar_sfull[t][bb]), (T >> 1) & 1, g, wait_code<37>());
        __syncwarp();
        tc_fence_after_sync();
        uint32_t ra[32], rb[32];
        tmem_ld32(s_col, ra);
        tmem_ld32(s_col + 32, rb);
        tmem_ld_wait(ra);
        reg_fence(rb);
        const int k0 = j * BK;
        if ((CAUSAL && (k0 + BK - 1 > q0t + p.off)) || (k0 + BK > p.Lk)) {
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            if (k0 + i > lim) ra[i] = __float_as_uint(-INFINITY);
            if (k0 + 32 + i > lim) rb[i] = __float_as_uint(-INFINITY);
          }
        }
        if (MASKED && !keep_t(pt, t, j)) {  // the other query tile needs this key tile
#pragma unroll
          for (int i = 0; i < 32; ++i) ra[i] = rb[i] = __float_as_uint(-INFINITY);
        }
        float mx[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) mx[i] = fmaxf(__uint_as_float(ra[i]), __uint_as_float(rb[i]));
#pragma unroll
        for (int i = 8; i < 32; ++i) mx[i & 7] = fmax3(mx[i & 7], __uint_as_float(ra[i]), __uint_as_float(rb[i]));
        const float mt = fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7])) * sl2;
        const float m_new = fmaxf(m, mt);
        if (__any_sync(0xffffffffu, m_new > m + Gm::TAU)) {
          const float alpha = ex2_approx(m - m_new);  // 0 on the first tile
          m = m_new;
          l *= alpha;
          if (k > 0) {
            // O_t holds P V up to the previous key tile once that MMA is done.
            // S_t of the next key tile was issued right after it, so its
            // barrier covers it; on the last key tile a dedicated commit does.
            if (k + 1 < nk)
              mbar_wait(smem_u32(&bar_sfull[t][(T + 1) & 1]), ((T + 1) >> 1) & 1, g, wait_code<39>());
            else
              mbar_wait(smem_u32(&bar_odone[t]), odone_ph, g, wait_code<40>());
            __syncwarp();
            tc_fence_after_sync();
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
              uint32_t rr[32];
              tmem_ld32(o_col + c * 32, rr);
              tmem_ld_wait(rr);
#pragma unroll
              for (int i = 0; i < 32; ++i) rr[i] = __float_as_uint(__uint_as_float(rr[i]) * alpha);
              tmem_st32(o_col + c * 32, rr);
            }
          }
        }
        // P = exp2(S * scale_log2 - m), two elements per packed instruction
        uint64_t sa2 = f2_pack(0.f, 0.f), sb2 = sa2;
        uint32_t pa[16], pb[16];
        // (a row that has seen no key yet keeps m = -inf and gets P = 0)
        const float mu = (MASKED && m == -INFINITY) ? 0.f : m;
        const uint64_t sl2x2 = f2_pack(sl2, sl2), nm2 = f2_pack(-mu, -mu);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          float x0, x1;
          f2_unpack(f2_fma(f2_pack(__uint_as_float(ra[2 * i]), __uint_as_float(ra[2 * i + 1])), sl2x2, nm2), x0, x1);
          const float a0 = ex2_approx(x0), a1 = ex2_approx(x1);
          f2_unpack(f2_fma(f2_pack(__uint_as_float(rb[2 * i]), __uint_as_float(rb[2 * i + 1])), sl2x2, nm2), x0, x1);
          const float b0 = ex2_approx(x0), b1 = ex2_approx(x1);
          sa2 = f2_add(sa2, f2_pack(a0, a1));
          sb2 = f2_add(sb2, f2_pack(b0, b1));
          pa[i] = E::pack(a0, a1);
          pb[i] = E::pack(b0, b1);
        }
        {
          float s0, s1, s2, s3;
          f2_unpack(sa2, s0, s1);
          f2_unpack(sb2, s2, s3);
          l += (s0 + s1) + (s2 + s3);
        }
        // P: keys 0..31 -> columns 0..15, keys 32..63 -> columns 16..31 of S_t
        tmem_st16(s_col, pa);
        tmem_st16(s_col + 16, pb);
        tmem_st_wait();
        tc_fence_before_sync();
        mbar_arrive(smem_u32(&bar_pready[t][bb]));
      }
      ts += nk;
      if (nk >= 2) odone_ph ^= 1u;
      // ---------------- epilogue ----------------
      mbar_wait(smem_u32(&bar_done), r & 1, g, wait_code<38>());
      __syncwarp();
      tc_fence_after_sync();
      const bool empty = MASKED && !(l > 0.f);  // the row saw no key: O = 0, lse = +inf
      const float inv_l = empty ? 0.f : 1.f / l;
      // O leaves through this warp's staging tile (its 32 rows x 64 columns
      // in the tensor map's swizzled layout) and one TMA store per 64
      // columns, which keeps the stores off the load/store unit: a store per
      // row from every thread would touch 32 rows' lines per instruction.
      // Rows past Lq are outside the map and are not written.
      const uint32_t stg = sO + warp * Gm::O_STG_BYTES;
#pragma unroll
      for (int h = 0; h < NCH; ++h) {
        // columns 64h .. 64h+63 (the second chunk exists unless D = 96, h = 1),
        // read and rounded while the tile's previous store still reads it
        const bool two = 2 * h + 1 < D / 32;
        uint32_t ra[32], rb[32], pa[16], pb[16];
        if (!MASKED || nk > 0) {  // same for the whole CTA: tcgen05.ld is warp-collective
          tmem_ld32(o_col + 2 * h * 32, ra);
          if (two) tmem_ld32(o_col + (2 * h + 1) * 32, rb);
          tmem_ld_wait(ra);  // waits for both loads
          if (two) reg_fence(rb);
        }
        if (MASKED && (nk == 0 || empty)) {
#pragma unroll
          for (int i = 0; i < 32; ++i) ra[i] = rb[i] = 0u;
        }
        pack_row32<BF16>(ra, inv_l, pa);
        if (two) pack_row32<BF16>(rb, inv_l, pb);
        if (lane == 0) bulk_wait_read_all();  // the tile's previous store has read it
        __syncwarp();
        stage_row16_sw128(stg + lane * 128, lane, 0, pa);
        if (two) stage_row16_sw128(stg + lane * 128, lane, 4, pb);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_3d(&tmO, stg, h * 64, q0t + quad * 32, bh);
          bulk_commit_group();
        }
      }
      if (qi < p.Lq && dbg_in_range(static_cast<size_t>(bh) * p.Lq + qi, 1, n_qrows, p.status, 2))
        p.lse[static_cast<size_t>(bh) * p.Lq + qi] = empty ? INFINITY : m + log2f(l);
      // the next item's first P V overwrites O_t after this warpgroup's next
      // P arrival, which follows these loads
      tc_fence_before_sync();
    }
    // the O stores have read their staging tiles and written global memory
    if (lane == 0) bulk_wait_all();
    __syncwarp();
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, Gm::TMEM_COLS);
  }
  if (threadIdx.x == 0) {
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
