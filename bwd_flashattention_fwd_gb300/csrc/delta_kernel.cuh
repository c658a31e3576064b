// delta_i = sum_d float(dO_id) * float(O_id), one float per query row
// ("feat(attention): complete Flash Attention VJP implementation", section
// "Two-Kernel Design": delta = rowsum(dO * O) in f32, computed once before the
// two gradient kernels).
//
// Purely bandwidth-bound: every input byte is read once, with coalesced loads.
// A row of D 16-bit elements is split across LPR consecutive lanes; each lane
// reads VEC bytes per load, the partial products are reduced with warp
// shuffles inside the LPR-lane group, and lane 0 of the group writes the row.
// Rows are handed out grid-stride, and each thread keeps UNROLL rows' loads in
// flight to cover HBM latency.
#pragma once

#include "kernel_common.cuh"

namespace gbattn {

template <int D>
struct DeltaGeom {
  // D = 96 rows (192 bytes) do not split into 16-byte pieces over a power-of-
  // two lane group, so they use 4-byte loads over 16 lanes (3 loads each).
  static constexpr int VEC = (D == 96) ? 4 : 16;  // bytes per load
  static constexpr int LPR = (D == 96) ? 16 : (D * 2) / 16;
  static constexpr int LOADS = (D * 2) / (VEC * LPR);
  static constexpr int ROWS_PER_WARP = 32 / LPR;
  static constexpr int UNROLL = 4;
  static constexpr int THREADS = 256;
  static_assert(LOADS * VEC * LPR == D * 2, "row split");
};

template <int VEC>
struct VecT;
template <>
struct VecT<16> {
  using T = uint4;
  static constexpr int WORDS = 4;
  __device__ __forceinline__ static T load(const void* p) {
    T v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
  }
  __device__ __forceinline__ static uint32_t word(const T& v, int i) {
    return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
  }
};
template <>
struct VecT<4> {
  using T = uint32_t;
  static constexpr int WORDS = 1;
  __device__ __forceinline__ static T load(const void* p) {
    T v;
    asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
  }
  __device__ __forceinline__ static uint32_t word(const T& v, int) { return v; }
};

template <int D, bool BF16>
__global__ void __launch_bounds__(256) attn_delta_kernel(const void* __restrict__ o,
                                                         const void* __restrict__ dO,
                                                         float* __restrict__ delta, long long rows) {
  using Gm = DeltaGeom<D>;
  using V = VecT<Gm::VEC>;
  using E = Elem<BF16>;
  // Launched behind the forward as a programmatic dependent: O is read only
  // once every earlier kernel on the stream has completed, and a dK/dV kernel
  // launched behind this one may start once every CTA of it has got here.
  grid_dependency_wait();
  if (threadIdx.x == 0) grid_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int sub = lane % Gm::LPR;        // lane within the row group
  const int grp = lane / Gm::LPR;        // row group within the warp
  const long long warp_global = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const long long n_warps = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
  const long long rows_per_step = n_warps * Gm::ROWS_PER_WARP;
  const char* ob = reinterpret_cast<const char*>(o);
  const char* db = reinterpret_cast<const char*>(dO);

  // The loop bound is uniform across the warp, so every shuffle sees all lanes.
  for (long long wbase = warp_global * Gm::ROWS_PER_WARP; wbase < rows;
       wbase += rows_per_step * Gm::UNROLL) {
    const long long base = wbase + grp;
    typename V::T ov[Gm::UNROLL][Gm::LOADS], dv[Gm::UNROLL][Gm::LOADS];
#pragma unroll
    for (int u = 0; u < Gm::UNROLL; ++u) {
      const long long row = base + u * rows_per_step;
      if (row < rows) {
#pragma unroll
        for (int l = 0; l < Gm::LOADS; ++l) {
          const long long off = row * (D * 2) + (l * Gm::LPR + sub) * Gm::VEC;
          ov[u][l] = V::load(ob + off);
          dv[u][l] = V::load(db + off);
        }
      }
    }
#pragma unroll
    for (int u = 0; u < Gm::UNROLL; ++u) {
      const long long row = base + u * rows_per_step;
      float acc = 0.f;
      if (row < rows) {
#pragma unroll
        for (int l = 0; l < Gm::LOADS; ++l)
#pragma unroll
          for (int w = 0; w < V::WORDS; ++w) {
            const float2 a = E::unpack(V::word(ov[u][l], w));
            const float2 c = E::unpack(V::word(dv[u][l], w));
            acc = fmaf(a.x, c.x, acc);
            acc = fmaf(a.y, c.y, acc);
          }
      }
#pragma unroll
      for (int sh = Gm::LPR / 2; sh > 0; sh >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, sh);
      if (sub == 0 && row < rows) delta[row] = acc;
    }
  }
}

}  // namespace gbattn
