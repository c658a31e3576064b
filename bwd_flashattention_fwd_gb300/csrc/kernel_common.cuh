// Definitions shared by the attention kernels: launch parameters, tile
// geometry, 16-bit packing and global stores.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "ptx.cuh"

namespace gbattn {

// Status codes a kernel may record in the device status word (the first
// nonzero code wins).  Values >= 100 identify which bounded wait ran out.
enum : int {
  kDevOk = 0,
  kDevTimeoutBase = 100,
};

constexpr uint64_t kDefaultWaitLimitNs = 2000000000ull;  // 2 s per wait
constexpr int kMaxDynSmem = 232448;                       // 227 KB per CTA on sm_103a
constexpr int kSmemReserve = 4096;                        // static shared memory

struct FwdParams {
  void* o;
  float* lse;
  int* status;
  int B, Hq, Hkv, Lq, Lk, G;
  int off;  // Lk - Lq: bottom-right causal offset
  int n_qtiles;
  float scale_log2;
  uint64_t limit_ns;
};

struct BwdParams {
  void* dq;
  void* dk;
  void* dv;
  const float* lse;
  const float* delta;
  int* status;
  int B, Hq, Hkv, Lq, Lk, G;
  int off;
  int n_qtiles, n_ktiles;  // in units of the launching kernel's own tiles
  float scale, scale_log2;
  uint64_t limit_ns;
};

template <bool BF16>
struct Elem;
template <>
struct Elem<true> {
  using T = __nv_bfloat16;
  __device__ __forceinline__ static uint32_t pack(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  }
  __device__ __forceinline__ static float2 unpack(uint32_t u) {
    __nv_bfloat162 v = *reinterpret_cast<__nv_bfloat162*>(&u);
    return __bfloat1622float2(v);
  }
};
template <>
struct Elem<false> {
  using T = __half;
  __device__ __forceinline__ static uint32_t pack(float lo, float hi) {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  }
  __device__ __forceinline__ static float2 unpack(uint32_t u) {
    __half2 v = *reinterpret_cast<__half2*>(&u);
    return __half22float2(v);
  }
};

// Number of 64-element (128-byte) column chunks a row of D 16-bit elements
// occupies in a 128-byte-swizzled tile.  D = 96 uses two chunks, the second
// half-filled with zeros by the TMA bounds.
__host__ __device__ constexpr int n_chunks(int D) { return (D + 63) / 64; }

// Scale 32 fp32 values and store them as 16-bit elements (64 bytes) to global
// memory at `dst` (16-byte aligned), as four 16-byte stores.
template <bool BF16>
__device__ __forceinline__ void store_row32(void* dst, const uint32_t (&r)[32], float mul) {
  uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint4 w;
    w.x = Elem<BF16>::pack(__uint_as_float(r[q * 8 + 0]) * mul, __uint_as_float(r[q * 8 + 1]) * mul);
    w.y = Elem<BF16>::pack(__uint_as_float(r[q * 8 + 2]) * mul, __uint_as_float(r[q * 8 + 3]) * mul);
    w.z = Elem<BF16>::pack(__uint_as_float(r[q * 8 + 4]) * mul, __uint_as_float(r[q * 8 + 5]) * mul);
    w.w = Elem<BF16>::pack(__uint_as_float(r[q * 8 + 6]) * mul, __uint_as_float(r[q * 8 + 7]) * mul);
    d[q] = w;
  }
}

// Position in a ring of N slots whose barriers flip phase once per lap:
// slot index and the parity of the current lap (cheaper than dividing a
// running tile count).
template <int N>
struct RingPos {
  int slot = 0;
  uint32_t phase = 0;
  __device__ __forceinline__ void next() {
    if (++slot == N) {
      slot = 0;
      phase ^= 1u;
    }
  }
};

}  // namespace gbattn
