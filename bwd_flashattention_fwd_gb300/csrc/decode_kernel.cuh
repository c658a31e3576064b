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

}  // namespace gbattn
