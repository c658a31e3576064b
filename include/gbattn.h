/*
 * gbattn -- exact causal grouped-query attention (forward with saved
 * log-sum-exp, delta precompute, fused two-kernel backward) for NVIDIA GB300
 * (sm_103a).  C ABI of libgbattn.so.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Pointers.  Every tensor pointer is a DEVICE pointer owned by the caller.
 *   The library never allocates per-call device memory and never frees caller
 *   memory.  Each pointer must be 16-byte aligned.
 * Layout.  Contiguous row-major [B, H, L, D]: D is the fastest axis, then the
 *   sequence position, then the head, then the batch.  q, o, dO, dq use
 *   H = Hq and L = Lq; k, v, dk, dv use H = Hkv and L = Lk.  lse and delta are
 *   float32 [B, Hq, Lq].  dq/dk/dv/o are written in the input dtype.
 * GQA.  Query head hq reads KV head hq / (Hq / Hkv): consecutive query heads
 *   share a KV head.
 * Causal alignment.  Bottom-right: key j is visible to query i iff
 *   j <= i + (Lk - Lq).  The offset comes from the true lengths ("Add a fused
 *   full-attention path for head_dim 256 on NAX devices", section "Ragged
 *   causal inputs").  Causal calls need Lk >= Lq, so every row sees a key.
 * Shapes.  B, Hq, Hkv, Lq, Lk >= 1; Hq % Hkv == 0; D in {64, 96, 128, 256}.
 *   Lq and Lk are arbitrary (ragged tails are masked inside the kernels).
 * Streams and errors.  Every call validates its arguments on the host first,
 *   without touching device memory, and returns ATTN_ERR_INVALID_ARG or
 *   ATTN_ERR_UNSUPPORTED before launching anything.  Otherwise it enqueues its
 *   kernels on `stream` and returns without synchronising; a launch failure
 *   returns ATTN_ERR_CUDA.  There is no fallback path: an unsupported shape is
 *   an error, never a silent change of implementation.  Device-side waits are
 *   bounded; a wait that runs out records ATTN_ERR_TIMEOUT in a device status
 *   word that attn_last_device_status() reports.
 * Debug build.  libgbattn_debug.so (the same sources compiled with
 *   GBATTN_DEBUG_CHECKS) checks every plain global load and store of its
 *   kernels against the extent of the tensor it addresses; an index outside
 *   is skipped, not performed, and recorded, so attn_last_device_status()
 *   returns ATTN_ERR_DEVICE_CHECK.  Nothing traps.  Same interface, same
 *   results, slower.
 */
#ifndef GBATTN_H_
#define GBATTN_H_

#include <cuda_runtime_api.h>
#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  ATTN_OK = 0,
  ATTN_ERR_INVALID_ARG = 1,
  ATTN_ERR_UNSUPPORTED = 2,
  ATTN_ERR_CUDA = 3,
  ATTN_ERR_TIMEOUT = 4,
  ATTN_ERR_DEVICE_CHECK = 5 /* debug build only: a kernel's index check failed */
} attn_status_t;

typedef enum { ATTN_DTYPE_FP16 = 0, ATTN_DTYPE_BF16 = 1 } attn_dtype_t;

/*
 * Forward with saved log-sum-exp.
 *   O = softmax(scale * Q K^T + mask) V, and per query row the base-2
 *   log-sum-exp lse_i = log2 sum_{j visible} exp2(scale * log2(e) * q_i.k_j).
 * Computed by an online softmax over key tiles ("When the Bottleneck Moved",
 * section 3, the running m / l / acc update and O = acc / l, L = m + log l),
 * in the log2 domain ("feat(attention): complete Flash Attention VJP
 * implementation", section "Background": P = exp2(S * scale_log2 - LSE)).
 *   q [B,Hq,Lq,D], k and v [B,Hkv,Lk,D]: inputs (dtype).
 *   o [B,Hq,Lq,D]: output (dtype).  lse [B,Hq,Lq]: output, float32, base 2.
 *   scale: finite and > 0 (usually 1/sqrt(D)).  causal: 0 or 1.
 */
attn_status_t attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                       int Hq, int Hkv, int Lq, int Lk, int D, float scale, int causal,
                       attn_dtype_t dtype, cudaStream_t stream);

/*
 * delta_i = sum_d float(dO_id) * float(O_id), float32 accumulation
 * ("feat(attention): complete Flash Attention VJP implementation", sections
 * "Reference implementation" and "Two-Kernel Design": delta = rowsum(dO * O)
 * computed once, before the two gradient kernels).
 *   o, dO [B,Hq,Lq,D]: inputs (dtype); o is the forward's stored output.
 *   delta [B,Hq,Lq]: output, float32.
 * Launched as a programmatic dependent of the work before it on the stream:
 * its CTAs may start while the previous kernel finishes, but it reads
 * nothing before all earlier work on the stream has completed, so stream
 * order holds for the caller as with a plain launch.  (The D <= 128 dK/dV
 * kernel of attn_bwd / attn_bwd_dkv is launched the same way.)
 */
attn_status_t attn_bwd_delta(const void* o, const void* dO, float* delta, int B, int Hq, int Lq,
                             int D, attn_dtype_t dtype, cudaStream_t stream);

/*
 * Fused backward: one dQ kernel (owns query rows, loops over key tiles) and
 * one dK/dV kernel (owns key rows, loops over the GQA group then query tiles),
 * so no output is shared and no atomics are needed ("feat(attention):
 * complete Flash Attention VJP implementation", sections "Background" and
 * "Two-Kernel Design").  Both recompute
 *   S = Q K^T,  P = exp2(S * scale * log2(e) - lse),  dP = dO V^T,
 *   dS = P * (dP - delta),
 * and accumulate dQ = scale * dS K, dK = scale * dS^T Q, dV = P^T dO.
 * The dQ kernel is launched behind the dK/dV kernel as a programmatic
 * dependent on the same stream, so it fills the SMs the dK/dV kernel's last
 * wave leaves idle; the call still completes as a whole in stream order.
 * Its CTAs take work from a counter in a per-device pool of 64 that calls
 * use in turn: at most 64 backward calls (attn_bwd, attn_bwd_dq and their
 * variants) may be in flight on one device at the same time.
 *   q, k, v, o, dO: inputs (dtype; o is accepted for interface symmetry and is
 *   only read through delta).  lse from attn_fwd and delta from attn_bwd_delta
 *   of the same (q, k, v, scale, causal): float32 [B,Hq,Lq].
 *   dq [B,Hq,Lq,D], dk and dv [B,Hkv,Lk,D]: outputs (dtype), fully overwritten.
 */
attn_status_t attn_bwd(const void* q, const void* k, const void* v, const void* o, const void* dO,
                       const float* lse, const float* delta, void* dq, void* dk, void* dv, int B,
                       int Hq, int Hkv, int Lq, int Lk, int D, float scale, int causal,
                       attn_dtype_t dtype, cudaStream_t stream);

/*
 * The two halves of attn_bwd, for callers that want to run them on different
 * streams (they share only read-only inputs, so they may run concurrently; the
 * pages' dQ and dK/dV kernels are encoded to run concurrently, "feat(attention):
 * complete Flash Attention VJP implementation", section "Two-Kernel Design").
 * attn_bwd(...) is exactly attn_bwd_dkv(...) followed by attn_bwd_dq(...) on
 * one stream.  Arguments as for attn_bwd; attn_bwd_dq writes only dq,
 * attn_bwd_dkv writes only dk and dv.
 */
attn_status_t attn_bwd_dq(const void* q, const void* k, const void* v, const void* dO, const float* lse,
                          const float* delta, void* dq, int B, int Hq, int Hkv, int Lq, int Lk, int D,
                          float scale, int causal, attn_dtype_t dtype, cudaStream_t stream);
attn_status_t attn_bwd_dkv(const void* q, const void* k, const void* v, const void* dO, const float* lse,
                           const float* delta, void* dk, void* dv, int B, int Hq, int Hkv, int Lq, int Lk,
                           int D, float scale, int causal, attn_dtype_t dtype, cudaStream_t stream);

/*
 * Block-sparse attention ("feat(attention): complete Flash Attention VJP
 * implementation", section "Sparse Block Masks": a uint8 entry per (query
 * tile, key tile) pair; a zero entry skips the pair).  These two calls are
 * attn_fwd and attn_bwd with a block mask on top of the causal mask:
 *   block_mask: DEVICE pointer, uint8, row-major [ceil(Lq/128), ceil(Lk/128)],
 *     shared by every batch and head; entry (qb, kb) != 0 keeps the pairs of
 *     query rows [128 qb, 128 qb + 128) and keys [128 kb, 128 kb + 128), 0
 *     removes them.  Owned by the caller, read only.
 *   Key tiles (forward, dQ) and query tiles (dK/dV) that the mask removes are
 *   neither loaded nor computed.  A query row left with no visible key gets
 *   O = 0 and lse = +inf (the pages do not define this case); its dQ is 0 and
 *   it adds nothing to dK and dV.  Feed attn_bwd_masked the lse of
 *   attn_fwd_masked with the same mask; delta comes from attn_bwd_delta.
 *   Every D of attn_fwd.  Other arguments and errors as for attn_fwd /
 *   attn_bwd; a null block_mask is ATTN_ERR_INVALID_ARG.
 */
attn_status_t attn_fwd_masked(const void* q, const void* k, const void* v, void* o, float* lse,
                              const uint8_t* block_mask, int B, int Hq, int Hkv, int Lq, int Lk, int D,
                              float scale, int causal, attn_dtype_t dtype, cudaStream_t stream);
attn_status_t attn_bwd_masked(const void* q, const void* k, const void* v, const void* o, const void* dO,
                              const float* lse, const float* delta, const uint8_t* block_mask, void* dq,
                              void* dk, void* dv, int B, int Hq, int Hkv, int Lq, int Lk, int D, float scale,
                              int causal, attn_dtype_t dtype, cudaStream_t stream);

/*
 * K and V sliced out of a longer key/value cache ("Add a fused full-attention
 * path for head_dim 256 on NAX devices", section "Ragged causal inputs": a
 * preallocated cache holds more positions per head than the call uses, so
 * the call's keys are keys[..., :Lk, :] of a [B, Hkv, capacity, D] buffer).
 * attn_fwd_ex / attn_bwd_ex are attn_fwd / attn_bwd with two options:
 *   block_mask: as for attn_fwd_masked, or NULL for no block mask.
 *   kv_pitch: rows between the starts of consecutive (b, hk) heads of k and v,
 *     i.e. the cache capacity; 0 means Lk (contiguous k and v).  Element
 *     (b, hk, j, d) of k is read at k + ((b*Hkv + hk)*kv_pitch + j)*D + d, for
 *     j < Lk only: rows j >= Lk of the cache (stale entries) are never read,
 *     whatever they hold.  dk and dv are written contiguous [B,Hkv,Lk,D].
 *   Errors: kv_pitch < 0 or 0 < kv_pitch < Lk is ATTN_ERR_INVALID_ARG; a pitch
 *   of 2^40 bytes or more per head is ATTN_ERR_UNSUPPORTED.  Everything else
 *   as for attn_fwd / attn_bwd.  Pass attn_bwd_ex the lse of attn_fwd_ex with the same options.
 */
attn_status_t attn_fwd_ex(const void* q, const void* k, const void* v, void* o, float* lse,
                          const uint8_t* block_mask, int64_t kv_pitch, int B, int Hq, int Hkv, int Lq,
                          int Lk, int D, float scale, int causal, attn_dtype_t dtype, cudaStream_t stream);
attn_status_t attn_bwd_ex(const void* q, const void* k, const void* v, const void* o, const void* dO,
                          const float* lse, const float* delta, const uint8_t* block_mask, int64_t kv_pitch,
                          void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int Lq, int Lk, int D,
                          float scale, int causal, attn_dtype_t dtype, cudaStream_t stream);

/*
 * Decode-shaped attention: short query lengths against long key ranges
 * ("feat(attention): complete Flash Attention VJP implementation": vector
 * kernels for sequences of at most 8; here any G * Lq <= 128, G = Hq / Hkv).
 * The same results as attn_fwd / attn_bwd (same arguments, layouts and
 * errors), computed for few query rows: the G query heads x Lq rows of each
 * KV head are processed as one tile of G*Lq rows, and each KV head's key
 * range is split over several CTAs whose partial results are merged.
 *   workspace: DEVICE pointer, 16-byte aligned, at least
 *     attn_decode_workspace_bytes(B, Hq, Hkv, Lq, Lk, D) bytes, owned by the
 *     caller; contents on entry are ignored and on exit are undefined.  One
 *     workspace may serve both calls but not two calls in flight at once.
 *   attn_decode_workspace_bytes returns 0 for a shape these calls reject
 *     (invalid, or G*Lq > 128).
 *   Errors: G*Lq > 128 is ATTN_ERR_UNSUPPORTED; a null, misaligned or too
 *   small workspace is ATTN_ERR_INVALID_ARG; the rest as for attn_fwd /
 *   attn_bwd.  attn_bwd_decode writes dk and dv with the attn_bwd_dkv kernel
 *   and dq with the split kernel; lse and delta as for attn_bwd (delta from
 *   attn_bwd_delta).
 */
size_t attn_decode_workspace_bytes(int B, int Hq, int Hkv, int Lq, int Lk, int D);
attn_status_t attn_fwd_decode(const void* q, const void* k, const void* v, void* o, float* lse, void* workspace,
                              size_t workspace_bytes, int B, int Hq, int Hkv, int Lq, int Lk, int D, float scale,
                              int causal, attn_dtype_t dtype, cudaStream_t stream);
attn_status_t attn_bwd_decode(const void* q, const void* k, const void* v, const void* o, const void* dO,
                              const float* lse, const float* delta, void* dq, void* dk, void* dv, void* workspace,
                              size_t workspace_bytes, int B, int Hq, int Hkv, int Lq, int Lk, int D, float scale,
                              int causal, attn_dtype_t dtype, cudaStream_t stream);

/*
 * attn_bwd for callers that cannot allocate device memory.  (The pages have no
 * counterpart: this is an entry point of this library only.)
 *
 * Who needs it: code whose device memory is fully managed by someone else --
 * a framework whose caching allocator already holds the GPU's memory, a
 * plugin whose execution callback must not allocate, a service that reserves
 * all memory at start-up and forbids allocation afterwards.  The other entry
 * points allocate one small device status word with cudaMalloc on their first
 * call on a device, and attn_bwd needs the caller to allocate delta; this one
 * needs neither.
 *
 * What it does: delta = rowsum(dO * O) (as attn_bwd_delta), then the dK/dV
 * and dQ kernels (as attn_bwd), with delta and the device status word kept in
 * a fixed scratch array that is part of the library image: 1 KB of header
 * (the status word and the dQ kernel's work counters) plus room for
 * B*Hq*Lq <= 1,048,576 delta values (4 MiB), held on
 * every GPU that loads the library until the process exits.  The call makes
 * no cudaMalloc, cudaFree or other allocating call.
 *   Arguments as for attn_bwd, without delta.  Larger problems (B*Hq*Lq above
 *   1,048,576) are rejected with ATTN_ERR_UNSUPPORTED before anything runs.
 *   Set-up: the first call on each device looks up the scratch array's device
 *   address (with that device current); make that first call before any
 *   stream capture.  A first call on a device made while `stream` is being
 *   captured is refused with ATTN_ERR_INVALID_ARG and changes nothing.
 *   Sharing: every call on a device uses the same scratch array, and the
 *   array keeps the last call's contents (the status word is cleared at the
 *   start of each call; delta is fully rewritten).  Calls whose work overlaps
 *   on the GPU -- on different streams without ordering between them -- race
 *   on the scratch and give wrong results; order them on one stream.
 *   Errors: argument and launch errors as for attn_bwd.  A bounded device wait
 *   that runs out is recorded in the scratch's status word, which
 *   attn_last_device_status reads and clears (reading it allocates nothing).
 */
attn_status_t attn_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const void* dO,
                               const float* lse, void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int Lq,
                               int Lk, int D, float scale, int causal, attn_dtype_t dtype, cudaStream_t stream);

/*
 * Synchronises `stream`, then reports and clears the device status words of the
 * current device (the one the entry points above share, and the one in
 * attn_bwd_noalloc's scratch): ATTN_ERR_TIMEOUT if a bounded device-side wait
 * ran out in a kernel since the last call, ATTN_ERR_DEVICE_CHECK if an index
 * check of the debug build failed, ATTN_ERR_CUDA if the stream reported an
 * error, ATTN_OK otherwise.  A failure is a typed error, never a
 * silent change of behaviour ("When the Bottleneck Moved", section 3: what
 * the implementation does not support fails with a typed error).
 */
attn_status_t attn_last_device_status(cudaStream_t stream);

/*
 * A check of the failure-reporting path; it computes nothing.  Launches one
 * CTA that waits, with the bounded wait every kernel of this library uses, on
 * an mbarrier that nothing ever completes.  When the wait limit runs out
 * (environment variable GBATTN_WAIT_LIMIT_NS, read once per process, in
 * nanoseconds; default 2 s) the wait records its code in the device status
 * word and the kernel returns, so the next attn_last_device_status(stream)
 * returns ATTN_ERR_TIMEOUT and the context stays usable.  Neither faults nor
 * hangs the GPU.  Returns ATTN_ERR_CUDA if the launch fails, else ATTN_OK.
 */
attn_status_t attn_wait_probe(cudaStream_t stream);

/* Static, human-readable name of a status code. */
const char* attn_status_string(attn_status_t s);

#ifdef __cplusplus
}
#endif

#endif /* GBATTN_H_ */
