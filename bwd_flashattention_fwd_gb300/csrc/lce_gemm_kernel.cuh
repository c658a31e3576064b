// The two gradient products of the linear cross-entropy backward ("When the
// Bottleneck Moved", section 1: the fused loss never forms the (N, V) logits;
// its backward recomputes one vocabulary chunk of g = dloss * (softmax -
// onehot) at a time, lce_kernel.cuh, and multiplies it out):
//   dH (+)= g W_chunk      C [tokens, hidden]     = A [tokens, chunk]  B [chunk, hidden]
//   dW_chunk = g^T H       C [chunk, hidden]      = A [chunk, tokens]  B [tokens, hidden]
//
// lce_gemm_kernel<BF16, A_MN> computes C = A B on the tensor cores in 128 x
// 256 tiles of C (tcgen05 MMAs, M = 128, N = 256, K = 16, fp32 accumulators
// in tensor memory), K in TMA stages of 64.  Both products read B with the
// hidden dimension contiguous, i.e. MN-major; A is K-major for dH (g rows are
// tokens, the chunk's vocabulary entries contiguous) and MN-major for dW (the
// same g memory read transposed), which A_MN selects.  Both operand layouts
// are the 128-byte-swizzled tiles a TMA load writes:
//   K-major   one box of 64 K-columns x 128 M-rows (rows 128 B apart);
//   MN-major  boxes of 64 MN-columns x 64 K-rows, one box per 64 MN-columns
//             (8 KB apart: the descriptor's leading-byte offset), rows 128 B
//             apart, 8-row groups 1 KB apart (its stride-byte offset).
// The epilogue (thread = row of the tile = TMEM lane) adds an optional fp32
// input and writes an fp32 result, a 16-bit result, or both, so dH can carry
// its fp32 sum from chunk to chunk and be rounded to 16 bits on the last one.
//
// Persistent CTAs (one per SM) walk the tiles with the hidden dimension
// innermost, so the CTAs in flight share their A rows and B columns through
// L2.  Two accumulators (2 x 256 TMEM columns) let one tile's epilogue run
// under the next tile's MMAs.  Warp roles (192 threads): warps 0-3 epilogue,
// warp 4 TMA producer, warp 5 MMA issuer and TMEM owner.
#pragma once

#include "kernel_common.cuh"

namespace gbattn {

struct LceGemmGeom {
  static constexpr int BM = 128;  // rows of C per tile: MMA M
  static constexpr int BN = 256;  // columns of C per tile: MMA N
  static constexpr int BK = 64;   // reduction length per stage
  static constexpr int A_BYTES = BM * BK * 2;
  static constexpr int B_BYTES = BN * BK * 2;
  static constexpr int MN_BOX_BYTES = 64 * BK * 2;  // one 64-column x 64-row MN-major box
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int STAGES = 4;
  static constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES;
  static constexpr int TMEM_COLS = 512;  // two accumulators of BN columns
  static constexpr int NUM_THREADS = 192;
  static_assert(SMEM_BYTES <= kMaxDynSmem - kSmemReserve, "shared memory budget");
};

struct LceGemmParams {
  int M, N;           // rows and columns of C that exist (N a multiple of 64)
  int n_mt, n_nt;     // tiles along M and N
  int n_kt;           // stages along K (the reduction length / 64, rounded up)
  int b_k0;           // B's row coordinate of K = 0 (the chunk start for W_chunk)
  const float* acc_in;  // [M][ldc] fp32 added to A B, or null
  float* acc_out;       // [M][ldc] fp32 result, or null
  void* out16;          // [M][ldc] 16-bit result, or null
  int ldc;
  int* status;
  uint64_t limit_ns;
};

// tmA: A_MN ? the [K rows][M columns] matrix, boxes 64 x 64
//           : the [M rows][K columns] matrix, boxes 64 x 128;
// tmB: the [K rows][N columns] matrix, boxes 64 x 64.
template <bool BF16, bool A_MN>
__global__ void __launch_bounds__(LceGemmGeom::NUM_THREADS, 1)
    lce_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const LceGemmParams p) {
  using Gm = LceGemmGeom;
  constexpr int BM = Gm::BM, BN = Gm::BN, BK = Gm::BK, ST = Gm::STAGES;

  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t bar_full[ST], bar_empty[ST], bar_accfull[2], bar_accempty[2];
  __shared__ uint32_t tmem_slot;
  __shared__ volatile int abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const int n_tiles = p.n_mt * p.n_nt;
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
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      tma_prefetch_desc(&tmA);
      tma_prefetch_desc(&tmB);
    }
    __syncwarp();
    RingPos<ST> st;
    int issued = 0;
    for (int t = blockIdx.x; t < n_tiles && !abort_flag; t += gridDim.x) {
      const int mt = t / p.n_nt, nt = t - mt * p.n_nt;
      const int m0 = mt * BM, n0 = nt * BN;
      for (int kt = 0; kt < p.n_kt; ++kt, st.next(), ++issued) {
        const int s = st.slot;
        if (issued >= ST) mbar_wait(smem_u32(&bar_empty[s]), st.phase ^ 1u, g, wait_code<51>());
        __syncwarp();
        if (abort_flag) break;  // after an abort no further copy is issued
        const uint32_t bar = smem_u32(&bar_full[s]);
        const uint32_t sA = sbase + s * Gm::STAGE_BYTES;
        const uint32_t sB = sA + Gm::A_BYTES;
        const int k0 = kt * BK;
        mbar_arrive_expect_tx_w(bar, Gm::STAGE_BYTES);
        if constexpr (A_MN) {
          tma_load_3d_w(sA, &tmA, bar, m0, k0, 0);
          tma_load_3d_w(sA + Gm::MN_BOX_BYTES, &tmA, bar, m0 + 64, k0, 0);
        } else {
          tma_load_3d_w(sA, &tmA, bar, k0, m0, 0);
        }
#pragma unroll
        for (int j = 0; j < BN / 64; ++j) tma_load_3d_w(sB + j * Gm::MN_BOX_BYTES, &tmB, bar, n0 + 64 * j, p.b_k0 + k0, 0);
      }
    }
    // the last ST issued stages (a stage is refilled only after its release,
    // so each holds at most one copy in flight) have landed before shared memory is released
    for (int u = 0; u < ST && u < issued; ++u) {
      if (st.slot == 0) st.phase ^= 1u;
      st.slot = (st.slot == 0 ? ST : st.slot) - 1;
      mbar_wait_drain(smem_u32(&bar_full[st.slot]), st.phase);
    }
    __syncwarp();
  } else if (warp == 5) {
    // ---------------- MMA issuer ----------------
    constexpr uint32_t IDESC = make_idesc_f16(BM, BN, BF16, A_MN, true);
    // K advances by 16 per MMA: 32 bytes along a K-major row, 16 rows (2 KB) of an MN-major box
    constexpr uint32_t A_KSTEP = A_MN ? 2048u : 32u;
    const uint64_t dA0 = A_MN ? make_sdesc_sw128(sbase, Gm::MN_BOX_BYTES, 1024) : make_sdesc_sw128(sbase, 16, 1024);
    const uint64_t dB0 = make_sdesc_sw128(sbase + Gm::A_BYTES, Gm::MN_BOX_BYTES, 1024);
    RingPos<ST> st;
    int u = 0;  // tiles of this CTA so far
    for (int t = blockIdx.x; t < n_tiles; t += gridDim.x, ++u) {
      const int b = u & 1;
      // the epilogue has read this accumulator's previous tile
      if (u >= 2) mbar_wait(smem_u32(&bar_accempty[b]), ((u >> 1) - 1) & 1, g, wait_code<52>());
      __syncwarp();
      tc_fence_after_sync();
      const uint32_t acc = tmem + b * BN;
      for (int kt = 0; kt < p.n_kt; ++kt, st.next()) {
        const int s = st.slot;
        mbar_wait(smem_u32(&bar_full[s]), st.phase, g, wait_code<53>());
        __syncwarp();
        tc_fence_after_sync();
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk)
          mma_ss_w(acc, sdesc_add(dA0, s * Gm::STAGE_BYTES + kk * A_KSTEP),
                   sdesc_add(dB0, s * Gm::STAGE_BYTES + kk * 2048u), IDESC, (kt > 0 || kk > 0) ? 1u : 0u);
        mma_commit_w(smem_u32(&bar_empty[s]));
      }
      mma_commit_w(smem_u32(&bar_accfull[b]));
    }
    // every MMA of the CTA is complete before tensor memory is released
    if (u > 0) mbar_wait_drain(smem_u32(&bar_accfull[(u - 1) & 1]), ((u - 1) >> 1) & 1);
    __syncwarp();
  } else {
    // ---------------- epilogue: thread = row of the tile ----------------
    using E = Elem<BF16>;
    const int r = warp * 32 + lane;
    const uint32_t lrow = static_cast<uint32_t>(warp * 32) << 16;
    int u = 0;
    for (int t = blockIdx.x; t < n_tiles; t += gridDim.x, ++u) {
      const int mt = t / p.n_nt, nt = t - mt * p.n_nt;
      const int b = u & 1;
      const int row = mt * BM + r;
      mbar_wait(smem_u32(&bar_accfull[b]), (u >> 1) & 1, g, wait_code<54>());
      __syncwarp();
      tc_fence_after_sync();
      const uint32_t acc = tmem + lrow + b * BN;
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c) {
        uint32_t rr[32];
        tmem_ld32(acc + c * 32, rr);
        tmem_ld_wait(rr);
        const int col = nt * BN + c * 32;
        if (row < p.M && col < p.N &&
            dbg_in_range(static_cast<size_t>(row) * p.ldc + col, 32, static_cast<size_t>(p.M) * p.ldc, p.status, 46)) {
          const size_t off = static_cast<size_t>(row) * p.ldc + col;
          if (p.acc_in) {
            const float4* src = reinterpret_cast<const float4*>(p.acc_in + off);
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              const float4 a = src[q];
              rr[4 * q + 0] = __float_as_uint(__uint_as_float(rr[4 * q + 0]) + a.x);
              rr[4 * q + 1] = __float_as_uint(__uint_as_float(rr[4 * q + 1]) + a.y);
              rr[4 * q + 2] = __float_as_uint(__uint_as_float(rr[4 * q + 2]) + a.z);
              rr[4 * q + 3] = __float_as_uint(__uint_as_float(rr[4 * q + 3]) + a.w);
            }
          }
          if (p.acc_out) store_row32_f32(p.acc_out + off, rr, 1.f);
          if (p.out16) store_row32<BF16>(static_cast<typename E::T*>(p.out16) + off, rr, 1.f);
        }
      }
      // accumulator read: the MMA warp may reuse it
      tc_fence_before_sync();
      mbar_arrive(smem_u32(&bar_accempty[b]));
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
