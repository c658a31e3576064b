// Definitions shared by the attention kernels: launch parameters, tile
// geometry, 16-bit packing and global stores.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "ptx.cuh"

namespace gbattn {

// Status codes a kernel may record in the device status word (the first
// nonzero code wins).  Values 100..199 identify which bounded wait ran out,
// values >= 200 which index check of a debug build failed.
enum : int {
  kDevOk = 0,
  kDevTimeoutBase = 100,
  kDevBoundsBase = 200,
};

// Status code of bounded wait number C of a kernel.  A template, so that a
// number that would leave the range of wait codes (and be read as a failed
// index check) does not compile.
template <int C>
__host__ __device__ constexpr int wait_code() {
  static_assert(C >= 1 && C < kDevBoundsBase - kDevTimeoutBase, "wait codes are 101..199");
  return kDevTimeoutBase + C;
}

// Debug build (compiled with -DGBATTN_DEBUG_CHECKS): every plain global load
// and store of the kernels first checks that the elements it touches,
// [first, first + count), lie inside the tensor's extent [0, extent).  A
// failed check records kDevBoundsBase + site in the status word and the
// access is skipped -- nothing traps, and the host reads the code through
// attn_last_device_status.  In the normal build the check is a constant
// `true` and compiles away.
#ifdef GBATTN_DEBUG_CHECKS
constexpr bool kDebugChecks = true;
#else
constexpr bool kDebugChecks = false;
#endif

__device__ __forceinline__ bool dbg_in_range(size_t first, size_t count, size_t extent, int* status, int site) {
  if constexpr (!kDebugChecks) {
    return true;
  } else {
    if (first + count <= extent && first + count >= first) return true;
    if (status) atomicCAS(status, 0, kDevBoundsBase + site);
    return false;
  }
}

constexpr uint64_t kDefaultWaitLimitNs = 2000000000ull;  // 2 s per wait
constexpr int kMaxDynSmem = 232448;                       // 227 KB per CTA on sm_103a
constexpr int kSmemReserve = 4096;                        // static shared memory
constexpr int kMaskBlock = 128;  // query rows and keys covered by one block-mask entry

struct FwdParams {
  void* o;
  float* lse;
  int* status;
  int B, Hq, Hkv, Lq, Lk, G;
  int off;  // Lk - Lq: bottom-right causal offset
  int n_qtiles;
  float scale_log2;
  uint64_t limit_ns;
  // block-sparse variant: uint8 [ceil(Lq/128), ceil(Lk/128)], row-major
  const uint8_t* bmask;
  int nkb;  // ceil(Lk / 128): row length of the mask
  // decode variant: Lq above is the packed row count G * Lq of one KV head,
  // qmod the true Lq (packed row r is query r % qmod); each CTA covers
  // split_tiles key tiles and writes fp32 partial O rows to ws and their
  // base-2 log-sum-exp to ws_lse
  int qmod, split_tiles;
  float* ws;
  float* ws_lse;
  // persistent forward: its work counter and the count of CTAs that have
  // finished (two ints, zero at launch; the last CTA puts them back to zero)
  int* sched;
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
  // block-sparse variant: uint8 [ceil(Lq/128), ceil(Lk/128)], row-major
  const uint8_t* bmask;
  int nkb;  // ceil(Lk / 128): row length of the mask
  int64_t kv_pitch;  // rows between consecutive heads of k and v (>= Lk)
  const void* k;     // K itself, for kernels that copy K rows into tensor memory
  const void* v;     // V itself, likewise
  // decode variant of the dQ kernel (as in FwdParams): fp32 partial dQ rows
  int qmod, split_tiles;
  float* ws;
  // persistent dQ kernel: its work counter and the count of CTAs that have
  // finished (two ints, zero at launch; the last CTA puts them back to zero)
  int* sched;
};

// fp32 row of 32 values (128 bytes, 16-byte aligned) to global memory, scaled.
__device__ __forceinline__ void store_row32_f32(float* dst, const uint32_t (&r)[32], float mul) {
  float4* d = reinterpret_cast<float4*>(dst);
#pragma unroll
  for (int q = 0; q < 8; ++q)
    d[q] = make_float4(__uint_as_float(r[4 * q]) * mul, __uint_as_float(r[4 * q + 1]) * mul,
                       __uint_as_float(r[4 * q + 2]) * mul, __uint_as_float(r[4 * q + 3]) * mul);
}

// Block-mask entry (query block qb, key block kb) of the launch parameters
// p (FwdParams or BwdParams); nonzero keeps the pair.
template <class Params>
__device__ __forceinline__ bool mask_keep(const Params& p, int qb, int kb) {
  const size_t i = static_cast<size_t>(qb) * p.nkb + kb;
  const size_t n = static_cast<size_t>((p.Lq + kMaskBlock - 1) / kMaskBlock) * p.nkb;
  return dbg_in_range(i, 1, n, p.status, 40) && __ldg(p.bmask + i) != 0;
}

// Walks the indices x in [lo, hi) for which keep(x) holds, in increasing
// order, testing 32 candidates per ballot.  Warp-collective: every lane calls
// first() and next() together and gets the same x; hi ends the walk.  Without
// a mask every index is kept and the walk is a plain count.
template <bool MASKED, class Keep>
struct KeptWalk {
  Keep keep;
  int hi;
  int base = 0;
  uint32_t bits = 0u;
  __device__ __forceinline__ int first(int lo) {
    if constexpr (!MASKED) {
      return lo;
    } else {
      base = lo - 32;
      bits = 0u;
      return next(lo - 1);
    }
  }
  __device__ __forceinline__ int next(int x) {
    if constexpr (!MASKED) {
      return x + 1;
    } else {
      while (bits == 0u) {
        base += 32;
        if (base >= hi) return hi;
        const int y = base + static_cast<int>(threadIdx.x & 31u);
        bits = __ballot_sync(0xffffffffu, y < hi && keep(y));
      }
      const int i = __ffs(static_cast<int>(bits)) - 1;
      bits &= bits - 1u;
      return base + i;
    }
  }
};

template <bool MASKED, class Keep>
__device__ __forceinline__ KeptWalk<MASKED, Keep> kept_walk(Keep keep, int hi) {
  return KeptWalk<MASKED, Keep>{keep, hi};
}

// Number of x in [lo, hi) with keep(x) (warp-collective).
template <bool MASKED, class Keep>
__device__ __forceinline__ int count_kept(Keep keep, int lo, int hi) {
  if (!MASKED) return hi - lo;
  int c = 0;
  for (int b = lo; b < hi; b += 32) {
    const int y = b + static_cast<int>(threadIdx.x & 31u);
    c += __popc(__ballot_sync(0xffffffffu, y < hi && keep(y)));
  }
  return c;
}

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
  __device__ __forceinline__ static T from_float(float x) { return __float2bfloat16_rn(x); }
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
  __device__ __forceinline__ static T from_float(float x) { return __float2half_rn(x); }
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

// Scale 32 fp32 values and round them to 16-bit pairs.
template <bool BF16>
__device__ __forceinline__ void pack_row32(const uint32_t (&v)[32], float mul, uint32_t (&pk)[16]) {
#pragma unroll
  for (int i = 0; i < 16; ++i)
    pk[i] = Elem<BF16>::pack(__uint_as_float(v[2 * i]) * mul, __uint_as_float(v[2 * i + 1]) * mul);
}

// Write 16 packed pairs (64 bytes) as the 16-byte pieces p0..p0+3 of row r of
// a shared-memory tile of 128-byte rows in the 128-byte-swizzled layout that
// a TMA store with that swizzle reads (piece p of row r sits (p ^ (r mod 8))
// * 16 bytes into the row; the tile starts on a 1024-byte boundary).  One
// warp writing one row per lane touches every bank group once per eight rows,
// so the four stores are free of conflicts.
__device__ __forceinline__ void stage_row16_sw128(uint32_t row_addr, int r, int p0, const uint32_t (&pk)[16]) {
#pragma unroll
  for (int q = 0; q < 4; ++q)
    st_shared_v4(row_addr + ((((p0 + q) ^ r) & 7) << 4), pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
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
