// The two small kernels that finish the decode-shaped (short query length)
// forward and dQ, which split each KV head's key range over several CTAs:
//
// attn_decode_combine_kernel merges the splits' partial results row by row
// with the online-softmax rule ("When the Bottleneck Moved", section 3): with
// partial base-2 log-sum-exps L_s and partial outputs O_s (each normalised by
// its own sum), M = max_s L_s, w_s = 2^(L_s - M), O = sum_s w_s O_s / sum_s w_s
// and lse = M + log2(sum_s w_s).
//
// attn_decode_dq_reduce_kernel sums the splits' fp32 shares of dS K and
// applies the softmax scale (dQ = scale * dS K, "feat(attention): complete
// Flash Attention VJP implementation", section "Background").
//
// Both are bound by memory traffic: one warp per output row (combine) or one
// thread per 4 output elements (reduce), fp32 partials read once.
#pragma once

#include "kernel_common.cuh"

namespace gbattn {

constexpr int kCombineThreads = 256;  // 8 rows per block

template <int D, bool BF16>
__global__ void __launch_bounds__(kCombineThreads)
    attn_decode_combine_kernel(const float* __restrict__ ws, const float* __restrict__ ws_lse, int n_split,
                               long long nrows, void* __restrict__ o, float* __restrict__ lse) {
  using E = Elem<BF16>;
  constexpr int PER = D / 32;  // columns per lane
  const long long row = static_cast<long long>(blockIdx.x) * (kCombineThreads / 32) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= nrows) return;
  float mx = -INFINITY;
  for (int s = 0; s < n_split; ++s) mx = fmaxf(mx, ws_lse[s * nrows + row]);
  float acc[PER];
#pragma unroll
  for (int c = 0; c < PER; ++c) acc[c] = 0.f;
  float den = 0.f;
  if (mx > -INFINITY) {
    for (int s = 0; s < n_split; ++s) {
      const float w = exp2f(ws_lse[s * nrows + row] - mx);  // 0 for a split that saw no key
      den += w;
      const float* src = ws + (s * nrows + row) * D;
#pragma unroll
      for (int c = 0; c < PER; ++c) acc[c] = fmaf(w, src[lane + 32 * c], acc[c]);
    }
  }
  // a row that saw no key at all (not reachable with causal Lq <= Lk): O = 0, lse = +inf
  const float inv = den > 0.f ? 1.f / den : 0.f;
  typename E::T* orow = reinterpret_cast<typename E::T*>(o) + row * D;
#pragma unroll
  for (int c = 0; c < PER; ++c) orow[lane + 32 * c] = E::from_float(acc[c] * inv);
  if (lane == 0) lse[row] = den > 0.f ? mx + log2f(den) : INFINITY;
}

constexpr int kReduceThreads = 256;

template <int D, bool BF16>
__global__ void __launch_bounds__(kReduceThreads)
    attn_decode_dq_reduce_kernel(const float* __restrict__ ws, int n_split, long long nrows, float scale,
                                 void* __restrict__ dq) {
  using E = Elem<BF16>;
  const long long n4 = nrows * D / 4;  // float4 groups
  for (long long i = static_cast<long long>(blockIdx.x) * kReduceThreads + threadIdx.x; i < n4;
       i += static_cast<long long>(gridDim.x) * kReduceThreads) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s = 0; s < n_split; ++s) {
      const float4 v = reinterpret_cast<const float4*>(ws)[s * n4 + i];
      acc.x += v.x, acc.y += v.y, acc.z += v.z, acc.w += v.w;
    }
    uint2 out;
    out.x = E::pack(acc.x * scale, acc.y * scale);
    out.y = E::pack(acc.z * scale, acc.w * scale);
    reinterpret_cast<uint2*>(dq)[i] = out;
  }
}

// ---------------------------------------------------------------------------
// Decode-shaped dK/dV (short query lengths, D <= 128).  The G query heads x Lq
// rows of a KV head form one packed tile of R <= 128 rows (row r is query
// r % Lq), and every key tile of the head meets that same tile, so each CTA
// loads the packed Q and dO tiles (and their lse / delta) once and streams a
// range of the head's 128-key tiles through a two-stage K/V ring.  Per key
// tile, with the key row as the TMEM lane (as in the general dK/dV kernel):
//   S^T = K Q^T, dP^T = V dO^T (N = 128 packed query columns; rows past R
//   have -lse = -inf and contribute nothing), P^T and dS^T from them,
//   dV = P^T dO and dK = dS^T Q accumulated over that one query tile,
// then dK, dV are read out and stored.  The next key tile's S^T and dP^T
// run while the row threads read the current tile's dK and dV out.
// ---------------------------------------------------------------------------
template <int D>
struct DecodeDkvGeom {
  static constexpr int BK = 128;  // keys per tile (MMA M)
  static constexpr int RQ = 128;  // packed query rows (MMA N of S^T)
  static constexpr int NCH = n_chunks(D);
  static constexpr int Q_BYTES = NCH * RQ * 128;  // a Q (or dO) tile
  static constexpr int KV_BYTES = NCH * BK * 128;  // a K (or V) tile
  static constexpr int STAGES = 2;
  static constexpr int SMEM_BYTES = 1024 + 2 * Q_BYTES + STAGES * 2 * KV_BYTES;
  static constexpr int ACC_W = 128;  // TMEM columns reserved for dK (and for dV)
  static constexpr int DK_COL = 0, DV_COL = ACC_W, ST_COL = 2 * ACC_W, DPT_COL = 2 * ACC_W + RQ;
  static constexpr int TMEM_COLS = 512;
  static constexpr int NUM_COMPUTE_WARPS = 8;
  static constexpr int NCT = 32 * NUM_COMPUTE_WARPS;
  static constexpr int PRODUCER_WARP = NUM_COMPUTE_WARPS;
  static constexpr int MMA_WARP = NUM_COMPUTE_WARPS + 1;
  static constexpr int NUM_THREADS = 32 * (NUM_COMPUTE_WARPS + 2);
  static_assert(D <= 128, "D <= 128");
  static_assert(DPT_COL + RQ <= TMEM_COLS, "tensor memory budget");
  static_assert(SMEM_BYTES <= kMaxDynSmem - kSmemReserve, "shared memory budget");
};

template <int D, bool BF16, bool CAUSAL>
__global__ void __launch_bounds__(DecodeDkvGeom<D>::NUM_THREADS, 1)
    attn_decode_dkv_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                           const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                           const BwdParams p) {
  using Gm = DecodeDkvGeom<D>;
  using E = Elem<BF16>;
  constexpr int BK = Gm::BK, RQ = Gm::RQ, NCH = Gm::NCH, ST = Gm::STAGES, NCT = Gm::NCT;
  // The split dQ kernel launched behind this one may start on the SMs this
  // grid frees as soon as every CTA of it is running (it reads none of its
  // outputs).
  if (threadIdx.x == 0) grid_launch_dependents();

  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t bar_q, bar_kvfull[ST], bar_kvempty[ST], bar_sfull, bar_pready, bar_accfull, bar_accfree,
      bar_mfin;
  __shared__ __align__(16) float nlse_s[RQ];  // -lse per packed query column (-inf past R)
  __shared__ __align__(16) float dlt_s[RQ];
  __shared__ uint32_t tmem_slot;
  __shared__ volatile int abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t sQ = sbase, sdO = sQ + Gm::Q_BYTES;
  const uint32_t sK0 = sdO + Gm::Q_BYTES;  // stage s: K at sK0 + 2 s KV_BYTES, V right after

  const int bhk = blockIdx.x;  // b * Hkv + hk: the packed tile's rows are bhk * R ..
  const int t0 = static_cast<int>(blockIdx.y) * p.split_tiles;
  const int n_t = min(p.n_ktiles - t0, p.split_tiles);  // key tiles t0 .. t0 + n_t - 1
  const WaitGuard g{&abort_flag, p.status, p.limit_ns};
  // extents for the debug build's index checks: rows of q / dq / lse /
  // delta, of dk / dv, and of the k / v buffers (pitch kv_pitch per head)
  [[maybe_unused]] const size_t n_qrows = static_cast<size_t>(p.B) * p.Hq * p.Lq;
  [[maybe_unused]] const size_t n_krows = static_cast<size_t>(p.B) * p.Hkv * p.Lk;
  [[maybe_unused]] const size_t n_kvbuf = (static_cast<size_t>(p.B) * p.Hkv - 1) * p.kv_pitch + p.Lk;

  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(smem_u32(&bar_q), 1 + 32);  // TMA expect_tx arrive + 32 producer lanes (lse / delta)
    for (int s = 0; s < ST; ++s) {
      mbar_init(smem_u32(&bar_kvfull[s]), 1);
      mbar_init(smem_u32(&bar_kvempty[s]), 1);
    }
    mbar_init(smem_u32(&bar_sfull), 1);
    mbar_init(smem_u32(&bar_pready), NCT);
    mbar_init(smem_u32(&bar_accfull), 1);
    mbar_init(smem_u32(&bar_accfree), NCT);
    mbar_init(smem_u32(&bar_mfin), 1);
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
      tma_prefetch_desc(&tmV);
      tma_prefetch_desc(&tmdO);
    }
    __syncwarp();
    mbar_arrive_expect_tx_w(smem_u32(&bar_q), 2 * Gm::Q_BYTES);
    for (int c = 0; c < NCH; ++c) {
      tma_load_3d_w(sQ + c * RQ * 128, &tmQ, smem_u32(&bar_q), c * 64, 0, bhk);
      tma_load_3d_w(sdO + c * RQ * 128, &tmdO, smem_u32(&bar_q), c * 64, 0, bhk);
    }
#pragma unroll
    for (int t = 0; t < RQ / 32; ++t) {
      const int c = lane + 32 * t;
      const size_t row = static_cast<size_t>(bhk) * p.Lq + c;
      nlse_s[c] = c < p.Lq && dbg_in_range(row, 1, n_qrows, p.status, 25) ? -p.lse[row] : -INFINITY;
      dlt_s[c] = c < p.Lq && dbg_in_range(row, 1, n_qrows, p.status, 26) ? p.delta[row] : 0.f;
    }
    mbar_arrive(smem_u32(&bar_q));
    int ni = 0;  // stages issued; after an abort (a wait ran out) no further copy is issued
    for (int i = 0; i < n_t; ++i) {
      const int s = i % ST;
      if (i >= ST) mbar_wait(smem_u32(&bar_kvempty[s]), (i / ST - 1) & 1, g, wait_code<58>());
      __syncwarp();
      if (abort_flag) break;
      ++ni;
      const uint32_t bar = smem_u32(&bar_kvfull[s]);
      const uint32_t dK = sK0 + 2 * s * Gm::KV_BYTES;
      mbar_arrive_expect_tx_w(bar, 2 * Gm::KV_BYTES);
      for (int c = 0; c < NCH; ++c) {
        tma_load_3d_w(dK + c * BK * 128, &tmK, bar, c * 64, (t0 + i) * BK, bhk);
        tma_load_3d_w(dK + Gm::KV_BYTES + c * BK * 128, &tmV, bar, c * 64, (t0 + i) * BK, bhk);
      }
    }
    // Q / dO and the last ST stages issued (a stage is refilled only after
    // its release, so each holds at most one copy in flight)
    mbar_wait_drain(smem_u32(&bar_q), 0);
    for (int i = (ni > ST ? ni - ST : 0); i < ni; ++i)
      mbar_wait_drain(smem_u32(&bar_kvfull[i % ST]), (i / ST) & 1);
  } else if (warp == Gm::MMA_WARP) {
    // ---------------- MMA issuer ----------------
    constexpr uint32_t IDESC_S = make_idesc_f16(128, RQ, BF16, false, false);
    constexpr uint32_t IDESC_ACC = make_idesc_f16(128, D, BF16, false, true);
    const uint64_t dKk = make_sdesc_sw128(sK0, 16, 1024);                 // K stage 0, K-major
    const uint64_t dVk = make_sdesc_sw128(sK0 + Gm::KV_BYTES, 16, 1024);  // V stage 0, K-major
    const uint64_t dQk = make_sdesc_sw128(sQ, 16, 1024);                  // Q, K-major
    const uint64_t dOk = make_sdesc_sw128(sdO, 16, 1024);                 // dO, K-major
    const uint64_t dQm = make_sdesc_sw128(sQ, RQ * 128, 1024);            // Q, MN-major
    const uint64_t dOm = make_sdesc_sw128(sdO, RQ * 128, 1024);           // dO, MN-major
    mbar_wait(smem_u32(&bar_q), 0, g, wait_code<59>());
    for (int i = 0; i < n_t; ++i) {
      const int s = i % ST;
      mbar_wait(smem_u32(&bar_kvfull[s]), (i / ST) & 1, g, wait_code<60>());
      __syncwarp();
      tc_fence_after_sync();
      // S^T and dP^T of key tile i; they overwrite P^T / dS^T of tile i-1
      // behind the dV / dK MMAs of tile i-1 that read them (issue order)
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t ko = 2 * s * Gm::KV_BYTES + (kk >> 2) * (BK * 128) + (kk & 3) * 32;
        const uint32_t qo = (kk >> 2) * (RQ * 128) + (kk & 3) * 32;
        mma_ss_w(tmem + Gm::ST_COL, sdesc_add(dKk, ko), sdesc_add(dQk, qo), IDESC_S, kk > 0 ? 1u : 0u);
        mma_ss_w(tmem + Gm::DPT_COL, sdesc_add(dVk, ko), sdesc_add(dOk, qo), IDESC_S, kk > 0 ? 1u : 0u);
      }
      mma_commit_w(smem_u32(&bar_sfull));
      mma_commit_w(smem_u32(&bar_kvempty[s]));  // K and V of the stage are read
      mbar_wait(smem_u32(&bar_pready), i & 1, g, wait_code<62>());
      // the row threads have read dK / dV of tile i-1 out
      if (i > 0) mbar_wait(smem_u32(&bar_accfree), (i - 1) & 1, g, wait_code<77>());
      __syncwarp();
      tc_fence_after_sync();
      // A operands: packed query columns 64h..64h+63 of warpgroup h sit as
      // pairs in columns 64h..64h+31 of the S^T (P^T) and dP^T (dS^T) buffers
#pragma unroll
      for (int kk = 0; kk < RQ / 16; ++kk) {
        const uint32_t acol = (kk >> 2) * 64 + (kk & 3) * 8;
        mma_ts_w(tmem + Gm::DV_COL, tmem + Gm::ST_COL + acol, sdesc_add(dOm, kk * 2048), IDESC_ACC,
                 kk > 0 ? 1u : 0u);
        mma_ts_w(tmem + Gm::DK_COL, tmem + Gm::DPT_COL + acol, sdesc_add(dQm, kk * 2048), IDESC_ACC,
                 kk > 0 ? 1u : 0u);
      }
      mma_commit_w(smem_u32(&bar_accfull));
    }
    // every MMA this warp issued is complete before tensor memory is released
    mma_commit_w(smem_u32(&bar_mfin));
    mbar_wait_drain(smem_u32(&bar_mfin), 0);
    __syncwarp();
  } else {
    // ---------------- key-row threads ----------------
    const int quad = warp & 3;   // TMEM lane quadrant (key rows)
    const int half = warp >> 2;  // packed query columns 64*half .. +63
    const int r = quad * 32 + lane;
    const uint32_t lrow = static_cast<uint32_t>(quad * 32) << 16;
    const uint64_t sl2x2 = f2_pack(p.scale_log2, p.scale_log2);
    mbar_wait(smem_u32(&bar_q), 0, g, wait_code<78>());  // the lse / delta tables
    for (int i = 0; i < n_t; ++i) {
      const int k0 = (t0 + i) * BK, kj = k0 + r;
      const int qmin = kj - p.off;  // causal: query indices below this cannot see key kj
      const bool need_mask = CAUSAL && (k0 + BK - 1 - p.off > 0);
      mbar_wait(smem_u32(&bar_sfull), i & 1, g, wait_code<79>());
      __syncwarp();
      tc_fence_after_sync();
#pragma unroll 1
      for (int cb = 0; cb < 2; ++cb) {  // two blocks of 32 packed query columns
        const int cc0 = half * 64 + cb * 32;
        const uint32_t scol = tmem + lrow + Gm::ST_COL + cc0, dcol = tmem + lrow + Gm::DPT_COL + cc0;
        uint32_t sr[32], dr[32];
        tmem_ld32(scol, sr);
        tmem_ld32(dcol, dr);
        tmem_ld_wait(sr);
        reg_fence(dr);
        const uint64_t* nlse_row = reinterpret_cast<const uint64_t*>(&nlse_s[cc0]);
        const uint64_t* dlt_row = reinterpret_cast<const uint64_t*>(&dlt_s[cc0]);
        int qq = cc0 % p.qmod;  // query index of packed column cc0
        uint32_t pk[16], dk[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int c0 = 2 * j;
          float x0, x1;
          f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[c0]), __uint_as_float(sr[c0 + 1])), sl2x2, nlse_row[j]), x0,
                    x1);
          float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
          if (need_mask) {
            if (qq < qmin) p0 = 0.f;
            qq = (qq + 1 == p.qmod) ? 0 : qq + 1;
            if (qq < qmin) p1 = 0.f;
            qq = (qq + 1 == p.qmod) ? 0 : qq + 1;
          }
          pk[j] = E::pack(p0, p1);
          const uint64_t d2 = f2_sub(f2_pack(__uint_as_float(dr[c0]), __uint_as_float(dr[c0 + 1])), dlt_row[j]);
          float ds0, ds1;
          f2_unpack(f2_mul(f2_pack(p0, p1), d2), ds0, ds1);
          dk[j] = E::pack(ds0, ds1);
        }
        // P^T / dS^T pairs of columns cc0..cc0+31 go to columns 64 half + 16 cb
        // .. +15: inside this warpgroup's own columns, over values it has read
        tmem_st16(tmem + lrow + Gm::ST_COL + half * 64 + cb * 16, pk);
        tmem_st16(tmem + lrow + Gm::DPT_COL + half * 64 + cb * 16, dk);
      }
      tmem_st_wait();
      tc_fence_before_sync();
      mbar_arrive(smem_u32(&bar_pready));
      // dK and dV of this key tile
      mbar_wait(smem_u32(&bar_accfull), i & 1, g, wait_code<80>());
      __syncwarp();
      tc_fence_after_sync();
      const size_t krow = static_cast<size_t>(bhk) * p.Lk + kj;
      typename E::T* dkrow = reinterpret_cast<typename E::T*>(p.dk) + krow * D;
      typename E::T* dvrow = reinterpret_cast<typename E::T*>(p.dv) + krow * D;
#pragma unroll 1
      for (int c = half; c < D / 32; c += 2) {
        uint32_t rr[32];
        tmem_ld32(tmem + lrow + Gm::DK_COL + c * 32, rr);
        tmem_ld_wait(rr);
        if (kj < p.Lk && dbg_in_range(krow * D + c * 32, 32, n_krows * D, p.status, 27))
          store_row32<BF16>(dkrow + c * 32, rr, p.scale);
        tmem_ld32(tmem + lrow + Gm::DV_COL + c * 32, rr);
        tmem_ld_wait(rr);
        if (kj < p.Lk && dbg_in_range(krow * D + c * 32, 32, n_krows * D, p.status, 28))
          store_row32<BF16>(dvrow + c * 32, rr, 1.f);
      }
      tc_fence_before_sync();
      mbar_arrive(smem_u32(&bar_accfree));
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == Gm::MMA_WARP) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, Gm::TMEM_COLS);
  }
}

}  // namespace gbattn
