// Linear cross-entropy without the (N, V) logits matrix ("When the Bottleneck
// Moved", section 1: logits = hidden @ W.T, loss_i = logsumexp(logits_i) -
// logits_i,target_i; the fused loss streams over vocabulary tiles, updates an
// online log-sum-exp, captures the target logit and returns per-token vectors).
//
// lce_logits_kernel computes 128 x 256 tiles of z = H W^T on the tensor cores
// (K = the hidden size, 64 columns per TMA stage, fp32 accumulators in tensor
// memory) and consumes each tile in its epilogue, so logits never reach
// global memory:
//   GRAD = false (forward): per row and vocabulary tile, the tile's maximum
//     m and sum s = sum_v 2^(z_v log2 e - m) (base 2), and the target's logit
//     when the tile holds it; lce_combine_kernel then merges the tiles of a
//     row into lse and loss (the online-softmax merge);
//   GRAD = true (backward): g = dloss * (exp(z - lse) - [v == target]) for one
//     chunk of the vocabulary, rounded to 16 bits and written out; the two
//     products dH += g W_chunk and dW_chunk = g^T H follow in
//     lce_gemm_kernel.cuh.
//
// Persistent CTAs walk the tiles vocabulary-major (all row tiles of a
// vocabulary tile, then the next), so the CTAs running at one time share a few
// W tiles through L2 and H stays in L2.  Two accumulator buffers (2 x 256
// TMEM columns) let the epilogue of one tile overlap the next tile's MMAs.
//
// Warp roles (192 threads): warps 0-3 epilogue (thread = row = TMEM lane),
// warp 4 TMA producer, warp 5 MMA issuer and TMEM owner.
#pragma once

#include "kernel_common.cuh"

namespace gbattn {

struct LceGeom {
  static constexpr int BM = 128;  // rows (tokens) per tile: MMA M
  static constexpr int BN = 256;  // vocabulary entries per tile: MMA N
  static constexpr int BK = 64;   // hidden columns per stage (one 128-byte swizzle row)
  static constexpr int A_BYTES = BM * 128;
  static constexpr int B_BYTES = BN * 128;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int STAGES = 4;
  static constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES;
  static constexpr int TMEM_COLS = 512;  // two accumulators of BN columns
  static constexpr int NUM_THREADS = 192;
  static_assert(SMEM_BYTES <= kMaxDynSmem - kSmemReserve, "shared memory budget");
};

struct LceParams {
  int N, Dm, V;
  int n_rt;   // row tiles: ceil(N / 128)
  int n_vt;   // vocabulary tiles of this launch
  int v0;     // first vocabulary entry of this launch (GRAD: the chunk start)
  int v_end;  // one past the last vocabulary entry of this launch
  const int* targets;
  // forward
  float2* part;      // [n_vt][N] (max, sum) per row and tile, base 2
  float* tgt_logit;  // [N]
  // backward
  const float* lse;    // [N], natural log
  const float* dloss;  // [N]
  void* g;             // [N][ldg] 16-bit, column 0 = vocabulary entry v0
  int ldg;
  int* status;
  uint64_t limit_ns;
};

template <bool BF16, bool GRAD>
__global__ void __launch_bounds__(LceGeom::NUM_THREADS, 1)
    lce_logits_kernel(const __grid_constant__ CUtensorMap tmH, const __grid_constant__ CUtensorMap tmW,
                      const LceParams p) {
  using Gm = LceGeom;
  using E = Elem<BF16>;
  constexpr int BM = Gm::BM, BN = Gm::BN, BK = Gm::BK, ST = Gm::STAGES;
  constexpr float kLog2e = 1.4426950408889634f;

  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t bar_full[ST], bar_empty[ST], bar_accfull[2], bar_accempty[2];
  __shared__ uint32_t tmem_slot;
  __shared__ volatile int abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const int n_tiles = p.n_vt * p.n_rt;
  const int nk = p.Dm / BK;
  const WaitGuard g{&abort_flag, p.status, p.limit_ns};

  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int s = 0; s < ST; ++s) {
      mbar_init(smem_u32(&bar_full[s]), 1);
      mbar_init(smem_u32(&bar_empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&bar_accfull[b]), 1);
      mbar_init(smem_u32(&bar_accempty[b]), 128);
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
      tma_prefetch_desc(&tmH);
      tma_prefetch_desc(&tmW);
    }
    __syncwarp();
    RingPos<ST> st;
    int issued = 0;
    for (int t = blockIdx.x; t < n_tiles && !abort_flag; t += gridDim.x) {
      const int vt = t / p.n_rt, rt = t - vt * p.n_rt;
      for (int k = 0; k < nk; ++k, st.next(), ++issued) {
        const int s = st.slot;
        if (issued >= ST) mbar_wait(smem_u32(&bar_empty[s]), st.phase ^ 1u, g, wait_code<41>());
        __syncwarp();
        if (abort_flag) break;  // after an abort no further copy is issued
        const uint32_t bar = smem_u32(&bar_full[s]);
        const uint32_t dA = sbase + s * Gm::STAGE_BYTES;
        mbar_arrive_expect_tx_w(bar, Gm::STAGE_BYTES);
        tma_load_3d_w(dA, &tmH, bar, k * BK, rt * BM, 0);
        tma_load_3d_w(dA + Gm::A_BYTES, &tmW, bar, k * BK, p.v0 + vt * BN, 0);
      }
    }
    // the last ST issued stages (a stage is refilled only after its release,
    // so each holds at most one copy in flight)
    for (int u = 0; u < ST && u < issued; ++u) {
      if (st.slot == 0) st.phase ^= 1u;
      st.slot = (st.slot == 0 ? ST : st.slot) - 1;
      mbar_wait_drain(smem_u32(&bar_full[st.slot]), st.phase);
    }
    __syncwarp();
  } else if (warp == 5) {
    // ---------------- MMA issuer ----------------
    constexpr uint32_t IDESC = make_idesc_f16(BM, BN, BF16, false, false);
    const uint64_t dA0 = make_sdesc_sw128(sbase, 16, 1024);                 // H stage 0, K-major
    const uint64_t dB0 = make_sdesc_sw128(sbase + Gm::A_BYTES, 16, 1024);  // W stage 0, K-major
    RingPos<ST> st;
    int u = 0;  // tiles of this CTA so far
    for (int t = blockIdx.x; t < n_tiles; t += gridDim.x, ++u) {
      const int b = u & 1;
      // the epilogue has read this accumulator's previous tile
      if (u >= 2) mbar_wait(smem_u32(&bar_accempty[b]), ((u >> 1) - 1) & 1, g, wait_code<42>());
      __syncwarp();
      tc_fence_after_sync();
      const uint32_t acc = tmem + b * BN;
      for (int k = 0; k < nk; ++k, st.next()) {
        const int s = st.slot;
        mbar_wait(smem_u32(&bar_full[s]), st.phase, g, wait_code<43>());
        __syncwarp();
        tc_fence_after_sync();
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk)
          mma_ss_w(acc, sdesc_add(dA0, s * Gm::STAGE_BYTES + kk * 32), sdesc_add(dB0, s * Gm::STAGE_BYTES + kk * 32),
                   IDESC, (k > 0 || kk > 0) ? 1u : 0u);
        mma_commit_w(smem_u32(&bar_empty[s]));
      }
      mma_commit_w(smem_u32(&bar_accfull[b]));
    }
    // every MMA of the CTA is complete before tensor memory is released
    if (u > 0) mbar_wait_drain(smem_u32(&bar_accfull[(u - 1) & 1]), ((u - 1) >> 1) & 1);
    __syncwarp();
  } else {
    // ---------------- epilogue: thread = row of the tile ----------------
    const int r = warp * 32 + lane;
    const uint32_t lrow = static_cast<uint32_t>(warp * 32) << 16;
    int u = 0;
    for (int t = blockIdx.x; t < n_tiles; t += gridDim.x, ++u) {
      const int vt = t / p.n_rt, rt = t - vt * p.n_rt;
      const int b = u & 1;
      const int row = rt * BM + r;
      const int tv0 = p.v0 + vt * BN;  // vocabulary entry of column 0
      const int n_valid = min(BN, p.v_end - tv0);
      const int tgt = row < p.N && dbg_in_range(row, 1, p.N, p.status, 41) ? p.targets[row] : -1;
      mbar_wait(smem_u32(&bar_accfull[b]), (u >> 1) & 1, g, wait_code<44>());
      __syncwarp();
      tc_fence_after_sync();
      const uint32_t acc = tmem + lrow + b * BN;
      if constexpr (!GRAD) {
        float m = -INFINITY, s = 0.f, zt = 0.f;
        const int tc = tgt - tv0;  // target's column in this tile, if 0 <= tc < n_valid
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          uint32_t rr[32];
          tmem_ld32(acc + c * 32, rr);
          tmem_ld_wait(rr);
          float y[32];
          float cm = -INFINITY;
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            y[i] = c * 32 + i < n_valid ? __uint_as_float(rr[i]) * kLog2e : -INFINITY;
            cm = fmaxf(cm, y[i]);
          }
          if (tc >= c * 32 && tc < c * 32 + 32 && tc < n_valid) {
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (tc == c * 32 + i) zt = __uint_as_float(rr[i]);
          }
          const float mn = fmaxf(m, cm);  // finite: column 0 of a tile is always valid
          float cs = 0.f;
#pragma unroll
          for (int i = 0; i < 32; ++i) cs += ex2_approx(y[i] - mn);
          s = s * ex2_approx(m - mn) + cs;
          m = mn;
        }
        // accumulator read: the MMA warp may reuse it
        tc_fence_before_sync();
        mbar_arrive(smem_u32(&bar_accempty[b]));
        if (row < p.N && dbg_in_range(static_cast<size_t>(vt) * p.N + row, 1, static_cast<size_t>(p.n_vt) * p.N,
                                      p.status, 42)) {
          p.part[static_cast<size_t>(vt) * p.N + row] = make_float2(m, s);
          if (tc >= 0 && tc < n_valid) p.tgt_logit[row] = zt;
        }
      } else {
        const float nl2 = row < p.N && dbg_in_range(row, 1, p.N, p.status, 43) ? -p.lse[row] * kLog2e : 0.f;
        const float d = (row < p.N && tgt >= 0 && tgt < p.V && dbg_in_range(row, 1, p.N, p.status, 44)) ? p.dloss[row]
                                                                                                     : 0.f;
        const int tc = tgt - tv0;
        typename E::T* grow = reinterpret_cast<typename E::T*>(p.g) +
                              static_cast<size_t>(row) * p.ldg + (tv0 - p.v0);
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          uint32_t rr[32];
          tmem_ld32(acc + c * 32, rr);
          tmem_ld_wait(rr);
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int c0 = c * 32 + 2 * i;
            float g0 = d * ex2_approx(fmaf(__uint_as_float(rr[2 * i]), kLog2e, nl2));
            float g1 = d * ex2_approx(fmaf(__uint_as_float(rr[2 * i + 1]), kLog2e, nl2));
            if (c0 == tc) g0 -= d;
            if (c0 + 1 == tc) g1 -= d;
            if (c0 >= n_valid) g0 = 0.f;
            if (c0 + 1 >= n_valid) g1 = 0.f;
            pk[i] = E::pack(g0, g1);
          }
          if (row < p.N && dbg_in_range(static_cast<size_t>(row) * p.ldg + (tv0 - p.v0) + c * 32, 32,
                                        static_cast<size_t>(p.N) * p.ldg, p.status, 45)) {
            uint4* dst = reinterpret_cast<uint4*>(grow + c * 32);
#pragma unroll
            for (int q = 0; q < 4; ++q) dst[q] = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
          }
        }
        tc_fence_before_sync();
        mbar_arrive(smem_u32(&bar_accempty[b]));
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

// Row-wise merge of the forward's tile partials: M = max_t m_t,
// lse = ln 2 * (M + log2 sum_t s_t 2^(m_t - M)), loss = lse - z_target
// (0 for a row whose target is negative or >= V: an ignored row).  One thread per row; the reads of a
// warp are consecutive rows of one tile's partials.
__global__ void __launch_bounds__(256)
    lce_combine_kernel(const float2* __restrict__ part, const float* __restrict__ tgt_logit,
                       const int* __restrict__ targets, int n_vt, int N, int V, float* __restrict__ loss,
                       float* __restrict__ lse) {
  const int row = blockIdx.x * 256 + threadIdx.x;
  if (row >= N) return;
  float M = -INFINITY;
  for (int t = 0; t < n_vt; ++t) M = fmaxf(M, part[static_cast<size_t>(t) * N + row].x);
  float S = 0.f;
  for (int t = 0; t < n_vt; ++t) {
    const float2 v = part[static_cast<size_t>(t) * N + row];
    S += v.y * exp2f(v.x - M);
  }
  const float l = (M + log2f(S)) * 0.69314718055994531f;
  lse[row] = l;
  const int t = targets[row];
  loss[row] = (t >= 0 && t < V) ? l - tgt_logit[row] : 0.f;
}

}  // namespace gbattn
