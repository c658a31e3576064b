// Host-side launch interface between the C ABI (api.cu) and the per-head-
// dimension kernel instantiations (inst.cu, compiled once per D).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

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
};

// Launch results: 0 = launched, 1 = tensor-map encoding rejected the
// arguments, 2 = CUDA launch error (cudaGetLastError() holds it).
enum LaunchResult : int { kLaunchOk = 0, kLaunchBadMap = 1, kLaunchCudaError = 2 };

#define GBATTN_DECLARE_LAUNCHERS(DIM)                \
  int launch_fwd_d##DIM(const AttnArgs& a);          \
  int launch_bwd_d##DIM(const AttnArgs& a);          \
  int launch_bwd_dq_d##DIM(const AttnArgs& a);       \
  int launch_bwd_dkv_d##DIM(const AttnArgs& a);      \
  int launch_delta_d##DIM(const AttnArgs& a);

GBATTN_DECLARE_LAUNCHERS(64)
GBATTN_DECLARE_LAUNCHERS(96)
GBATTN_DECLARE_LAUNCHERS(128)
GBATTN_DECLARE_LAUNCHERS(256)

#undef GBATTN_DECLARE_LAUNCHERS

}  // namespace gbattn
