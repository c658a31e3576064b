// Host-side launch interface between the C ABI (api.cu) and the per-head-
// dimension kernel instantiations (inst.cu, compiled once per D).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/gbattn.h"

namespace gbattn {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// Everything one call needs; pointers are device pointers owned by the caller.
struct AttnArgs {
  const void* q = nullptr;
  const void* k = nullptr;
  const void* v = nullptr;
  const void* o = nullptr;
  const void* dO = nullptr;
  const float* lse = nullptr;
  const float* delta = nullptr;
  void* o_out = nullptr;
  float* lse_out = nullptr;
  float* delta_out = nullptr;
  void* dq = nullptr;
  void* dk = nullptr;
  void* dv = nullptr;
  int B = 0, Hq = 0, Hkv = 0, Lq = 0, Lk = 0, D = 0;
  float scale = 0.f;
  bool causal = false;
  bool bf16 = true;
  cudaStream_t stream = nullptr;
  int* status = nullptr;  // device status word
  uint64_t limit_ns = 0;
  int num_sms = 0;
  EncodeTiledFn encode = nullptr;
  // block-sparse variant: uint8 [ceil(Lq/128), ceil(Lk/128)] on the device, or null
  const uint8_t* block_mask = nullptr;
  // rows between consecutive (b, hk) heads of k and v; 0 = Lk (contiguous)
  int64_t kv_pitch = 0;
  // decode calls: caller's fp32 workspace (see decode_layout)
  float* workspace = nullptr;
  // the persistent dQ kernel's work counter: two ints in device memory, zero
  // between launches (one slot of the library's per-device pool)
  int* sched = nullptr;
  // the dQ launch follows the dK/dV launch on the same stream and may run
  // beside its last wave (programmatic dependent launch)
  bool dq_behind_dkv = false;
};

// Decode-shaped calls (G * Lq <= 128): each KV head's G query heads x Lq rows
// form one packed tile, and its key range is split over several CTAs, about
// kDecodeCtas in all (two waves on a 152-SM GB300), at least one key tile
// each.  The forward's partials take n_split x rows x (D + 1) floats, the
// dQ kernel's n_split x rows x D floats, rows = B * Hq * Lq.
constexpr int kDecodeCtas = 304;
constexpr int kDecodeMaxRows = 128;

struct DecodeSplit {
  int tiles_per_split;
  int n_split;
};

inline DecodeSplit decode_split(long long groups, int n_tiles) {
  long long n = (kDecodeCtas + groups - 1) / groups;
  if (n > n_tiles) n = n_tiles;
  if (n < 1) n = 1;
  const int per = static_cast<int>((n_tiles + n - 1) / n);
  return {per, (n_tiles + per - 1) / per};
}

// key tiles of the forward (128 keys, 64 at D = 256) and dQ (64 keys) kernels
inline int decode_fwd_tiles(int Lk, int D) { return (Lk + (D <= 128 ? 128 : 64) - 1) / (D <= 128 ? 128 : 64); }
inline int decode_dq_tiles(int Lk) { return (Lk + 63) / 64; }

inline size_t decode_workspace_bytes(int B, int Hkv, long long rows, int Lk, int D) {
  const long long groups = static_cast<long long>(B) * Hkv;
  const DecodeSplit f = decode_split(groups, decode_fwd_tiles(Lk, D));
  const DecodeSplit q = decode_split(groups, decode_dq_tiles(Lk));
  const size_t fb = static_cast<size_t>(f.n_split) * rows * (D + 1) * 4;
  const size_t qb = static_cast<size_t>(q.n_split) * rows * D * 4;
  return fb > qb ? fb : qb;
}

// Device state shared by every call of the library (api.cu): tensor-map
// encoder, device status word, SM count; and the bounded-wait limit.
attn_status_t shared_device_state(int* dev, EncodeTiledFn* enc, int** status, int* num_sms);
uint64_t shared_wait_limit_ns();

// Launch results: 0 = launched, 1 = tensor-map encoding rejected the
// arguments, 2 = CUDA launch error (cudaGetLastError() holds it).
enum LaunchResult : int { kLaunchOk = 0, kLaunchBadMap = 1, kLaunchCudaError = 2 };

#define GBATTN_DECLARE_LAUNCHERS(DIM)                \
  int launch_fwd_d##DIM(const AttnArgs& a);          \
  int launch_bwd_d##DIM(const AttnArgs& a);          \
  int launch_bwd_dq_d##DIM(const AttnArgs& a);       \
  int launch_bwd_dkv_d##DIM(const AttnArgs& a);      \
  int launch_delta_d##DIM(const AttnArgs& a);       \
  int launch_fwd_decode_d##DIM(const AttnArgs& a);   \
  int launch_bwd_dkv_decode_d##DIM(const AttnArgs& a); \
  int launch_bwd_dq_decode_d##DIM(const AttnArgs& a);

GBATTN_DECLARE_LAUNCHERS(64)
GBATTN_DECLARE_LAUNCHERS(96)
GBATTN_DECLARE_LAUNCHERS(128)
GBATTN_DECLARE_LAUNCHERS(256)

#undef GBATTN_DECLARE_LAUNCHERS

}  // namespace gbattn
