// C ABI of libgbattn.so (declared in include/gbattn.h): argument validation,
// the per-device status word, and dispatch to the per-head-dimension
// launchers.  Validation is synchronous and touches no device memory.
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <mutex>

#include "../../include/gbattn.h"
#include "kernel_common.cuh"
#include "launch.h"

namespace gbattn {
namespace {

constexpr int kMaxDevices = 64;

std::mutex g_mu;
EncodeTiledFn g_encode = nullptr;
int* g_status[kMaxDevices] = {};
int g_num_sms[kMaxDevices] = {};

// Work counters of the persistent forward (D <= 128) and dQ kernels:
// kSchedSlots pairs of ints per device, zero between launches (each launch's
// last CTA resets its pair).  Calls take the slots in turn, so calls in
// flight at the same time on one device use different counters unless more
// than kSchedSlots of them overlap.
constexpr int kSchedSlots = 64;
int* g_sched[kMaxDevices] = {};
std::atomic<unsigned> g_sched_next[kMaxDevices];

int* sched_slot(int* pool, std::atomic<unsigned>& next) {
  return pool + 2 * (next.fetch_add(1u, std::memory_order_relaxed) % kSchedSlots);
}

uint64_t wait_limit_ns() {
  static const uint64_t v = [] {
    const char* s = std::getenv("GBATTN_WAIT_LIMIT_NS");
    if (s && *s) {
      const unsigned long long x = std::strtoull(s, nullptr, 10);
      if (x > 0) return static_cast<uint64_t>(x);
    }
    return static_cast<uint64_t>(2000000000ull);
  }();
  return v;
}

// Per-device state created on first use: the tensor-map encoder (a driver
// entry point), the device status word (one int, zeroed) and the SM count.
attn_status_t device_state(int* dev_out, EncodeTiledFn* enc, int** status, int* num_sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn)
      return ATTN_ERR_CUDA;
    g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  }
  if (!g_status[dev]) {
    int* p = nullptr;
    if (cudaMalloc(&p, sizeof(int)) != cudaSuccess) return ATTN_ERR_CUDA;
    if (cudaMemset(p, 0, sizeof(int)) != cudaSuccess) return ATTN_ERR_CUDA;
    int* sp = nullptr;
    if (cudaMalloc(&sp, 2 * kSchedSlots * sizeof(int)) != cudaSuccess) return ATTN_ERR_CUDA;
    if (cudaMemset(sp, 0, 2 * kSchedSlots * sizeof(int)) != cudaSuccess) return ATTN_ERR_CUDA;
    g_sched[dev] = sp;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return ATTN_ERR_CUDA;
    g_num_sms[dev] = sms;
    g_status[dev] = p;
  }
  *dev_out = dev;
  *enc = g_encode;
  *status = g_status[dev];
  *num_sms = g_num_sms[dev];
  return ATTN_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool supported_d(int D) { return D == 64 || D == 96 || D == 128 || D == 256; }

attn_status_t check_common(int B, int Hq, int Lq, int D, attn_dtype_t dtype) {
  if (B <= 0 || Hq <= 0 || Lq <= 0) return ATTN_ERR_INVALID_ARG;
  if (dtype != ATTN_DTYPE_FP16 && dtype != ATTN_DTYPE_BF16) return ATTN_ERR_INVALID_ARG;
  if (!supported_d(D)) return ATTN_ERR_UNSUPPORTED;
  // grid limits: B*H CTAs along x, 64-row tiles along y
  if (static_cast<long long>(B) * Hq > 0x7fffffffLL) return ATTN_ERR_UNSUPPORTED;
  if ((Lq + 63) / 64 > 65535) return ATTN_ERR_UNSUPPORTED;
  // work items of the persistent dQ kernel (128-row query tiles x heads)
  if (static_cast<long long>(B) * Hq * ((Lq + 127) / 128) > 0x7fffffffLL) return ATTN_ERR_UNSUPPORTED;
  return ATTN_OK;
}

attn_status_t check_attention(int B, int Hq, int Hkv, int Lq, int Lk, int D, float scale, int causal,
                              attn_dtype_t dtype) {
  const attn_status_t s = check_common(B, Hq, Lq, D, dtype);
  if (s == ATTN_ERR_INVALID_ARG) return s;
  if (Hkv <= 0 || Lk <= 0) return ATTN_ERR_INVALID_ARG;
  if (Hq % Hkv != 0) return ATTN_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return ATTN_ERR_INVALID_ARG;
  if (causal && Lq > Lk) return ATTN_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.f)) return ATTN_ERR_INVALID_ARG;
  if (s != ATTN_OK) return s;
  if ((Lk + 63) / 64 > 65535) return ATTN_ERR_UNSUPPORTED;
  return ATTN_OK;
}

attn_status_t finish(int r) {
  if (r == kLaunchOk) return ATTN_OK;
  if (r == kLaunchBadMap) return ATTN_ERR_INVALID_ARG;
  return ATTN_ERR_CUDA;
}

int dispatch_fwd(const AttnArgs& a) {
  switch (a.D) {
    case 64: return launch_fwd_d64(a);
    case 96: return launch_fwd_d96(a);
    case 128: return launch_fwd_d128(a);
    default: return launch_fwd_d256(a);
  }
}
int dispatch_bwd(const AttnArgs& a) {
  switch (a.D) {
    case 64: return launch_bwd_d64(a);
    case 96: return launch_bwd_d96(a);
    case 128: return launch_bwd_d128(a);
    default: return launch_bwd_d256(a);
  }
}
int dispatch_bwd_dq(const AttnArgs& a) {
  switch (a.D) {
    case 64: return launch_bwd_dq_d64(a);
    case 96: return launch_bwd_dq_d96(a);
    case 128: return launch_bwd_dq_d128(a);
    default: return launch_bwd_dq_d256(a);
  }
}
int dispatch_bwd_dkv(const AttnArgs& a) {
  switch (a.D) {
    case 64: return launch_bwd_dkv_d64(a);
    case 96: return launch_bwd_dkv_d96(a);
    case 128: return launch_bwd_dkv_d128(a);
    default: return launch_bwd_dkv_d256(a);
  }
}
int dispatch_fwd_decode(const AttnArgs& a) {
  switch (a.D) {
    case 64: return launch_fwd_decode_d64(a);
    case 96: return launch_fwd_decode_d96(a);
    case 128: return launch_fwd_decode_d128(a);
    default: return launch_fwd_decode_d256(a);
  }
}
int dispatch_bwd_dkv_decode(const AttnArgs& a) {
  switch (a.D) {
    case 64: return launch_bwd_dkv_decode_d64(a);
    case 96: return launch_bwd_dkv_decode_d96(a);
    case 128: return launch_bwd_dkv_decode_d128(a);
    default: return launch_bwd_dkv_decode_d256(a);
  }
}
int dispatch_bwd_dq_decode(const AttnArgs& a) {
  switch (a.D) {
    case 64: return launch_bwd_dq_decode_d64(a);
    case 96: return launch_bwd_dq_decode_d96(a);
    case 128: return launch_bwd_dq_decode_d128(a);
    default: return launch_bwd_dq_decode_d256(a);
  }
}
int dispatch_delta(const AttnArgs& a) {
  switch (a.D) {
    case 64: return launch_delta_d64(a);
    case 96: return launch_delta_d96(a);
    case 128: return launch_delta_d128(a);
    default: return launch_delta_d256(a);
  }
}

// Row pitch of k and v: 0 (contiguous) or at least Lk, within the TMA
// stride limit (2^40 bytes between heads).
attn_status_t check_kv_pitch(int64_t kv_pitch, int Lk, int D) {
  if (kv_pitch < 0 || (kv_pitch != 0 && kv_pitch < Lk)) return ATTN_ERR_INVALID_ARG;
  if (kv_pitch > (int64_t{1} << 40) / (2 * D)) return ATTN_ERR_UNSUPPORTED;
  return ATTN_OK;
}

// Forward with an optional block mask (null = none) and K/V row pitch.
attn_status_t fwd_call(const void* q, const void* k, const void* v, void* o, float* lse, const uint8_t* block_mask,
                       int64_t kv_pitch, int B, int Hq, int Hkv, int Lq, int Lk, int D, float scale, int causal,
                       attn_dtype_t dtype, cudaStream_t stream) {
  if (!q || !k || !v || !o || !lse) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return ATTN_ERR_INVALID_ARG;
  attn_status_t s = check_attention(B, Hq, Hkv, Lq, Lk, D, scale, causal, dtype);
  if (s != ATTN_OK) return s;
  s = check_kv_pitch(kv_pitch, Lk, D);
  if (s != ATTN_OK) return s;
  AttnArgs a;
  int dev;
  const attn_status_t ds = device_state(&dev, &a.encode, &a.status, &a.num_sms);
  if (ds != ATTN_OK) return ds;
  a.q = q, a.k = k, a.v = v, a.o_out = o, a.lse_out = lse, a.block_mask = block_mask, a.kv_pitch = kv_pitch;
  a.sched = sched_slot(g_sched[dev], g_sched_next[dev]);
  a.B = B, a.Hq = Hq, a.Hkv = Hkv, a.Lq = Lq, a.Lk = Lk, a.D = D;
  a.scale = scale, a.causal = causal != 0, a.bf16 = dtype == ATTN_DTYPE_BF16;
  a.stream = stream, a.limit_ns = wait_limit_ns();
  return finish(dispatch_fwd(a));
}

// Backward (dK/dV kernel, then dQ kernel) with the same options.
attn_status_t bwd_call(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse,
                       const float* delta, const uint8_t* block_mask, int64_t kv_pitch, void* dq, void* dk, void* dv,
                       int B, int Hq, int Hkv, int Lq, int Lk, int D, float scale, int causal, attn_dtype_t dtype,
                       cudaStream_t stream) {
  if (!q || !k || !v || !o || !dO || !lse || !delta || !dq || !dk || !dv) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(dO) || !aligned16(dq) || !aligned16(dk) ||
      !aligned16(dv))
    return ATTN_ERR_INVALID_ARG;
  attn_status_t s = check_attention(B, Hq, Hkv, Lq, Lk, D, scale, causal, dtype);
  if (s != ATTN_OK) return s;
  s = check_kv_pitch(kv_pitch, Lk, D);
  if (s != ATTN_OK) return s;
  AttnArgs a;
  int dev;
  const attn_status_t ds = device_state(&dev, &a.encode, &a.status, &a.num_sms);
  if (ds != ATTN_OK) return ds;
  a.q = q, a.k = k, a.v = v, a.o = o, a.dO = dO, a.lse = lse, a.delta = delta;
  a.block_mask = block_mask, a.kv_pitch = kv_pitch;
  a.dq = dq, a.dk = dk, a.dv = dv;
  a.sched = sched_slot(g_sched[dev], g_sched_next[dev]);
  a.B = B, a.Hq = Hq, a.Hkv = Hkv, a.Lq = Lq, a.Lk = Lk, a.D = D;
  a.scale = scale, a.causal = causal != 0, a.bf16 = dtype == ATTN_DTYPE_BF16;
  a.stream = stream, a.limit_ns = wait_limit_ns();
  return finish(dispatch_bwd(a));
}

// Decode calls: the packed tile (G * Lq rows) must fit 128 rows, and the
// caller's workspace must hold the split partials.
attn_status_t check_decode(int B, int Hq, int Hkv, int Lq, int Lk, int D, const void* ws, size_t ws_bytes) {
  if (static_cast<long long>(Hq / Hkv) * Lq > kDecodeMaxRows) return ATTN_ERR_UNSUPPORTED;
  if (!ws || !aligned16(ws)) return ATTN_ERR_INVALID_ARG;
  const long long rows = static_cast<long long>(B) * Hq * Lq;
  if (ws_bytes < decode_workspace_bytes(B, Hkv, rows, Lk, D)) return ATTN_ERR_INVALID_ARG;
  return ATTN_OK;
}

}  // namespace
}  // namespace gbattn

namespace gbattn {
// For the other translation units of the library (the linear cross-entropy
// calls share the device state and the status word).
attn_status_t shared_device_state(int* dev, EncodeTiledFn* enc, int** status, int* num_sms) {
  return device_state(dev, enc, status, num_sms);
}
uint64_t shared_wait_limit_ns() { return wait_limit_ns(); }
}  // namespace gbattn

using namespace gbattn;

extern "C" attn_status_t attn_bwd_delta(const void* o, const void* dO, float* delta, int B, int Hq, int Lq, int D,
                                        attn_dtype_t dtype, cudaStream_t stream) {
  if (!o || !dO || !delta) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(o) || !aligned16(dO) || !aligned16(delta)) return ATTN_ERR_INVALID_ARG;
  const attn_status_t s = check_common(B, Hq, Lq, D, dtype);
  if (s != ATTN_OK) return s;
  AttnArgs a;
  int dev;
  const attn_status_t ds = device_state(&dev, &a.encode, &a.status, &a.num_sms);
  if (ds != ATTN_OK) return ds;
  a.o = o, a.dO = dO, a.delta_out = delta;
  a.B = B, a.Hq = Hq, a.Hkv = Hq, a.Lq = Lq, a.Lk = Lq, a.D = D;
  a.bf16 = dtype == ATTN_DTYPE_BF16, a.stream = stream;
  return finish(dispatch_delta(a));
}

extern "C" attn_status_t attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
                                  int Hkv, int Lq, int Lk, int D, float scale, int causal, attn_dtype_t dtype,
                                  cudaStream_t stream) {
  return fwd_call(q, k, v, o, lse, nullptr, 0, B, Hq, Hkv, Lq, Lk, D, scale, causal, dtype, stream);
}

extern "C" attn_status_t attn_bwd(const void* q, const void* k, const void* v, const void* o, const void* dO,
                                  const float* lse, const float* delta, void* dq, void* dk, void* dv, int B, int Hq,
                                  int Hkv, int Lq, int Lk, int D, float scale, int causal, attn_dtype_t dtype,
                                  cudaStream_t stream) {
  return bwd_call(q, k, v, o, dO, lse, delta, nullptr, 0, dq, dk, dv, B, Hq, Hkv, Lq, Lk, D, scale, causal, dtype,
                  stream);
}

// Block-sparse variants: the same calls with a [ceil(Lq/128), ceil(Lk/128)]
// uint8 block mask on the device.
extern "C" attn_status_t attn_fwd_masked(const void* q, const void* k, const void* v, void* o, float* lse,
                                         const uint8_t* block_mask, int B, int Hq, int Hkv, int Lq, int Lk, int D,
                                         float scale, int causal, attn_dtype_t dtype, cudaStream_t stream) {
  if (!block_mask) return ATTN_ERR_INVALID_ARG;
  return fwd_call(q, k, v, o, lse, block_mask, 0, B, Hq, Hkv, Lq, Lk, D, scale, causal, dtype, stream);
}

extern "C" attn_status_t attn_bwd_masked(const void* q, const void* k, const void* v, const void* o,
                                         const void* dO, const float* lse, const float* delta,
                                         const uint8_t* block_mask, void* dq, void* dk, void* dv, int B, int Hq,
                                         int Hkv, int Lq, int Lk, int D, float scale, int causal, attn_dtype_t dtype,
                                         cudaStream_t stream) {
  if (!block_mask) return ATTN_ERR_INVALID_ARG;
  return bwd_call(q, k, v, o, dO, lse, delta, block_mask, 0, dq, dk, dv, B, Hq, Hkv, Lq, Lk, D, scale, causal,
                  dtype, stream);
}

// Every option at once: an optional block mask (null = none) and the row
// pitch of k and v (0 = Lk, i.e. contiguous; larger when they are the first
// Lk rows of each head of a longer cache).
extern "C" attn_status_t attn_fwd_ex(const void* q, const void* k, const void* v, void* o, float* lse,
                                     const uint8_t* block_mask, int64_t kv_pitch, int B, int Hq, int Hkv, int Lq,
                                     int Lk, int D, float scale, int causal, attn_dtype_t dtype, cudaStream_t stream) {
  return fwd_call(q, k, v, o, lse, block_mask, kv_pitch, B, Hq, Hkv, Lq, Lk, D, scale, causal, dtype, stream);
}

extern "C" attn_status_t attn_bwd_ex(const void* q, const void* k, const void* v, const void* o, const void* dO,
                                     const float* lse, const float* delta, const uint8_t* block_mask,
                                     int64_t kv_pitch, void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int Lq,
                                     int Lk, int D, float scale, int causal, attn_dtype_t dtype, cudaStream_t stream) {
  return bwd_call(q, k, v, o, dO, lse, delta, block_mask, kv_pitch, dq, dk, dv, B, Hq, Hkv, Lq, Lk, D, scale,
                  causal, dtype, stream);
}

// Decode-shaped attention (short query lengths, "feat(attention): complete
// Flash Attention VJP implementation": the vector kernels for L <= 8).
extern "C" size_t attn_decode_workspace_bytes(int B, int Hq, int Hkv, int Lq, int Lk, int D) {
  if (check_attention(B, Hq, Hkv, Lq, Lk, D, 1.f, 0, ATTN_DTYPE_BF16) != ATTN_OK) return 0;
  if (static_cast<long long>(Hq / Hkv) * Lq > kDecodeMaxRows) return 0;
  return decode_workspace_bytes(B, Hkv, static_cast<long long>(B) * Hq * Lq, Lk, D);
}

extern "C" attn_status_t attn_fwd_decode(const void* q, const void* k, const void* v, void* o, float* lse,
                                         void* workspace, size_t workspace_bytes, int B, int Hq, int Hkv, int Lq,
                                         int Lk, int D, float scale, int causal, attn_dtype_t dtype,
                                         cudaStream_t stream) {
  if (!q || !k || !v || !o || !lse) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return ATTN_ERR_INVALID_ARG;
  attn_status_t s = check_attention(B, Hq, Hkv, Lq, Lk, D, scale, causal, dtype);
  if (s != ATTN_OK) return s;
  s = check_decode(B, Hq, Hkv, Lq, Lk, D, workspace, workspace_bytes);
  if (s != ATTN_OK) return s;
  AttnArgs a;
  int dev;
  const attn_status_t ds = device_state(&dev, &a.encode, &a.status, &a.num_sms);
  if (ds != ATTN_OK) return ds;
  a.q = q, a.k = k, a.v = v, a.o_out = o, a.lse_out = lse, a.workspace = static_cast<float*>(workspace);
  a.B = B, a.Hq = Hq, a.Hkv = Hkv, a.Lq = Lq, a.Lk = Lk, a.D = D;
  a.scale = scale, a.causal = causal != 0, a.bf16 = dtype == ATTN_DTYPE_BF16;
  a.stream = stream, a.limit_ns = wait_limit_ns();
  return finish(dispatch_fwd_decode(a));
}

extern "C" attn_status_t attn_bwd_decode(const void* q, const void* k, const void* v, const void* o, const void* dO,
                                         const float* lse, const float* delta, void* dq, void* dk, void* dv,
                                         void* workspace, size_t workspace_bytes, int B, int Hq, int Hkv, int Lq,
                                         int Lk, int D, float scale, int causal, attn_dtype_t dtype,
                                         cudaStream_t stream) {
  if (!q || !k || !v || !o || !dO || !lse || !delta || !dq || !dk || !dv) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(dO) || !aligned16(dq) || !aligned16(dk) ||
      !aligned16(dv))
    return ATTN_ERR_INVALID_ARG;
  attn_status_t s = check_attention(B, Hq, Hkv, Lq, Lk, D, scale, causal, dtype);
  if (s != ATTN_OK) return s;
  s = check_decode(B, Hq, Hkv, Lq, Lk, D, workspace, workspace_bytes);
  if (s != ATTN_OK) return s;
  AttnArgs a;
  int dev;
  const attn_status_t ds = device_state(&dev, &a.encode, &a.status, &a.num_sms);
  if (ds != ATTN_OK) return ds;
  a.q = q, a.k = k, a.v = v, a.o = o, a.dO = dO, a.lse = lse, a.delta = delta, a.dq = dq, a.dk = dk, a.dv = dv;
  a.workspace = static_cast<float*>(workspace);
  a.B = B, a.Hq = Hq, a.Hkv = Hkv, a.Lq = Lq, a.Lk = Lk, a.D = D;
  a.scale = scale, a.causal = causal != 0, a.bf16 = dtype == ATTN_DTYPE_BF16;
  a.stream = stream, a.limit_ns = wait_limit_ns();
  const int r = dispatch_bwd_dkv_decode(a);
  a.dq_behind_dkv = true;
  return finish(r == kLaunchOk ? dispatch_bwd_dq_decode(a) : r);
}

// The two halves of attn_bwd, for callers that run them on separate streams.
namespace {
attn_status_t bwd_part(bool dq_part, const void* q, const void* k, const void* v, const void* dO,
                       const float* lse, const float* delta, void* dq, void* dk, void* dv, int B, int Hq, int Hkv,
                       int Lq, int Lk, int D, float scale, int causal, attn_dtype_t dtype, cudaStream_t stream) {
  if (!q || !k || !v || !dO || !lse || !delta) return ATTN_ERR_INVALID_ARG;
  if (dq_part ? !dq : (!dk || !dv)) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(dO)) return ATTN_ERR_INVALID_ARG;
  if (dq_part ? !aligned16(dq) : (!aligned16(dk) || !aligned16(dv))) return ATTN_ERR_INVALID_ARG;
  const attn_status_t s = check_attention(B, Hq, Hkv, Lq, Lk, D, scale, causal, dtype);
  if (s != ATTN_OK) return s;
  AttnArgs a;
  int dev;
  const attn_status_t ds = device_state(&dev, &a.encode, &a.status, &a.num_sms);
  if (ds != ATTN_OK) return ds;
  a.q = q, a.k = k, a.v = v, a.dO = dO, a.lse = lse, a.delta = delta;
  a.dq = dq, a.dk = dk, a.dv = dv;
  a.sched = sched_slot(g_sched[dev], g_sched_next[dev]);
  a.B = B, a.Hq = Hq, a.Hkv = Hkv, a.Lq = Lq, a.Lk = Lk, a.D = D;
  a.scale = scale, a.causal = causal != 0, a.bf16 = dtype == ATTN_DTYPE_BF16;
  a.stream = stream, a.limit_ns = wait_limit_ns();
  return finish(dq_part ? dispatch_bwd_dq(a) : dispatch_bwd_dkv(a));
}
}  // namespace

extern "C" attn_status_t attn_bwd_dq(const void* q, const void* k, const void* v, const void* dO, const float* lse,
                                     const float* delta, void* dq, int B, int Hq, int Hkv, int Lq, int Lk, int D,
                                     float scale, int causal, attn_dtype_t dtype, cudaStream_t stream) {
  return bwd_part(true, q, k, v, dO, lse, delta, dq, nullptr, nullptr, B, Hq, Hkv, Lq, Lk, D, scale, causal, dtype,
                  stream);
}

extern "C" attn_status_t attn_bwd_dkv(const void* q, const void* k, const void* v, const void* dO,
                                      const float* lse, const float* delta, void* dk, void* dv, int B, int Hq,
                                      int Hkv, int Lq, int Lk, int D, float scale, int causal, attn_dtype_t dtype,
                                      cudaStream_t stream) {
  return bwd_part(false, q, k, v, dO, lse, delta, nullptr, dk, dv, B, Hq, Hkv, Lq, Lk, D, scale, causal, dtype,
                  stream);
}

// ---------------------------------------------------------------------------
// attn_bwd_noalloc: the backward for callers that cannot allocate device
// memory.  Its scratch (the device status word and the delta vector) lives in
// the static array below instead of in memory obtained from cudaMalloc.
// ---------------------------------------------------------------------------
namespace {

constexpr long long kNoAllocMaxRows = 1LL << 20;  // B * Hq * Lq, i.e. 4 MiB of delta
// header: the status word at 0, the dQ kernel's work counters at 256
// (kSchedSlots pairs of ints, zero between launches), padded to 1 KB
constexpr size_t kNoAllocSchedOffset = 256;
constexpr size_t kNoAllocHeaderBytes = 1024;
static_assert(kNoAllocSchedOffset + 2 * kSchedSlots * sizeof(int) <= kNoAllocHeaderBytes, "scratch header");
constexpr size_t kNoAllocBytes = kNoAllocHeaderBytes + sizeof(float) * static_cast<size_t>(kNoAllocMaxRows);

// Loaded with the library on every GPU that uses it, and kept until exit.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocBytes];

std::mutex g_noalloc_mu;
EncodeTiledFn g_noalloc_encode = nullptr;
unsigned char* g_noalloc_ptr[kMaxDevices] = {};
int g_noalloc_sms[kMaxDevices] = {};
std::atomic<unsigned> g_noalloc_sched_next[kMaxDevices];

// Once per device, with that device current: the device address of the
// scratch array (host code only sees a stand-in for the symbol), the SM count
// and the tensor-map encoder.  None of these calls allocates device memory.
attn_status_t noalloc_setup(int* dev_out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn)
      return ATTN_ERR_CUDA;
    g_noalloc_encode = reinterpret_cast<EncodeTiledFn>(fn);
  }
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return ATTN_ERR_CUDA;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return ATTN_ERR_CUDA;
    g_noalloc_sms[dev] = sms;
    g_noalloc_ptr[dev] = static_cast<unsigned char*>(p);
  }
  *dev_out = dev;
  return ATTN_OK;
}

// Whether the device's scratch address has been looked up already.
bool noalloc_ready() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  return g_noalloc_ptr[dev] != nullptr;
}

// The scratch's status word on the current device, or null before set-up.
int* noalloc_status_word(int dev) {
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  return g_noalloc_ptr[dev] ? reinterpret_cast<int*>(g_noalloc_ptr[dev]) : nullptr;
}

}  // namespace

extern "C" attn_status_t attn_bwd_noalloc(const void* q, const void* k, const void* v, const void* o,
                                          const void* dO, const float* lse, void* dq, void* dk, void* dv, int B,
                                          int Hq, int Hkv, int Lq, int Lk, int D, float scale, int causal,
                                          attn_dtype_t dtype, cudaStream_t stream) {
  if (!q || !k || !v || !o || !dO || !lse || !dq || !dk || !dv) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(dO) || !aligned16(dq) ||
      !aligned16(dk) || !aligned16(dv))
    return ATTN_ERR_INVALID_ARG;
  const attn_status_t s = check_attention(B, Hq, Hkv, Lq, Lk, D, scale, causal, dtype);
  if (s != ATTN_OK) return s;
  if (static_cast<long long>(B) * Hq * Lq > kNoAllocMaxRows) return ATTN_ERR_UNSUPPORTED;
  // The first call on a device looks the scratch address up, which may load
  // the module: not allowed while the stream is being captured.
  if (!noalloc_ready()) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone) {
      cudaGetLastError();  // an implicit-capture error must not linger for later calls
      return ATTN_ERR_INVALID_ARG;
    }
  }
  int dev = 0;
  const attn_status_t ss = noalloc_setup(&dev);
  if (ss != ATTN_OK) return ss;
  unsigned char* scratch = g_noalloc_ptr[dev];
  int* status = reinterpret_cast<int*>(scratch);
  float* dlt = reinterpret_cast<float*>(scratch + kNoAllocHeaderBytes);
  // The status word must start each call at zero; delta is fully rewritten.
  if (cudaMemsetAsync(status, 0, sizeof(int), stream) != cudaSuccess) return ATTN_ERR_CUDA;
  AttnArgs a;
  a.encode = g_noalloc_encode;
  a.num_sms = g_noalloc_sms[dev];
  a.status = status;
  a.q = q, a.k = k, a.v = v, a.o = o, a.dO = dO, a.lse = lse, a.delta = dlt, a.delta_out = dlt;
  a.dq = dq, a.dk = dk, a.dv = dv;
  a.sched = sched_slot(reinterpret_cast<int*>(scratch + kNoAllocSchedOffset), g_noalloc_sched_next[dev]);
  a.B = B, a.Hq = Hq, a.Hkv = Hkv, a.Lq = Lq, a.Lk = Lk, a.D = D;
  a.scale = scale, a.causal = causal != 0, a.bf16 = dtype == ATTN_DTYPE_BF16;
  a.stream = stream, a.limit_ns = wait_limit_ns();
  const int r = dispatch_delta(a);
  if (r != kLaunchOk) return finish(r);
  return finish(dispatch_bwd(a));
}

// ---------------------------------------------------------------------------
// attn_wait_probe: a check of the failure-reporting path.  One CTA waits,
// with the same bounded wait as every kernel of the library, on an mbarrier
// that nothing ever completes; when the wait limit runs out the wait records
// its code in the status word and returns, and the kernel ends.
// ---------------------------------------------------------------------------
namespace gbattn {
namespace probe {

constexpr int kProbeCode = wait_code<99>();

__global__ void attn_wait_probe_kernel(int* status, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  __shared__ volatile int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(smem_u32(&bar), 1);  // one arrival expected; none is ever made
    fence_mbar_init();
  }
  __syncthreads();
  const WaitGuard g{&abort_flag, status, limit_ns};
  mbar_wait(smem_u32(&bar), 0, g, kProbeCode);
  __syncthreads();
}

// Reads the status word at `p` (device memory) into *code and clears it;
// false on a CUDA error.  Neither call allocates.
bool take_status_word(int* p, int* code) {
  *code = 0;
  if (cudaMemcpy(code, p, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return false;
  return *code == 0 || cudaMemset(p, 0, sizeof(int)) == cudaSuccess;
}

}  // namespace probe
}  // namespace gbattn

extern "C" attn_status_t attn_wait_probe(cudaStream_t stream) {
  int dev, num_sms, *status;
  EncodeTiledFn enc;
  const attn_status_t ds = device_state(&dev, &enc, &status, &num_sms);
  if (ds != ATTN_OK) return ds;
  probe::attn_wait_probe_kernel<<<1, 32, 0, stream>>>(status, wait_limit_ns());
  return cudaPeekAtLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

extern "C" attn_status_t attn_last_device_status(cudaStream_t stream) {
  if (cudaStreamSynchronize(stream) != cudaSuccess) return ATTN_ERR_CUDA;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
  int* p;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    p = g_status[dev];
  }
  // the allocating entry points' word, then the word in attn_bwd_noalloc's
  // scratch; a failed index check (debug build) outranks a timeout
  attn_status_t st = ATTN_OK;
  for (int* w : {p, noalloc_status_word(dev)}) {
    int code = 0;
    if (!w) continue;
    if (!probe::take_status_word(w, &code)) return ATTN_ERR_CUDA;
    if (code >= kDevBoundsBase) st = ATTN_ERR_DEVICE_CHECK;
    else if (code != 0 && st == ATTN_OK) st = ATTN_ERR_TIMEOUT;
  }
  return st;
}

extern "C" const char* attn_status_string(attn_status_t s) {
  switch (s) {
    case ATTN_OK: return "ATTN_OK";
    case ATTN_ERR_INVALID_ARG: return "ATTN_ERR_INVALID_ARG";
    case ATTN_ERR_UNSUPPORTED: return "ATTN_ERR_UNSUPPORTED";
    case ATTN_ERR_CUDA: return "ATTN_ERR_CUDA";
    case ATTN_ERR_TIMEOUT: return "ATTN_ERR_TIMEOUT";
    case ATTN_ERR_DEVICE_CHECK: return "ATTN_ERR_DEVICE_CHECK";
    default: return "ATTN_ERR_UNKNOWN";
  }
}
