/*
 * gblce -- linear cross-entropy without the (N, V) logits matrix, for NVIDIA
 * GB300 (sm_103a).  Part of libgbattn.so; status and dtype codes, pointer
 * conventions and attn_last_device_status() are those of gbattn.h.
 *
 * What it computes ("When the Bottleneck Moved", section 1 "The first
 * hypothesis: remove logits, train longer": logits = hidden @ W.T,
 * loss_i = logsumexp(logits_i) - logits_i,target_i, with the fused loss
 * streaming over vocabulary tiles, updating an online log-sum-exp, capturing
 * the target logit and returning only per-token vectors):
 *   forward   loss[i] = lse[i] - z[i, t[i]],  lse[i] = log sum_v exp z[i, v],
 *             z = hidden @ weight^T (never stored);
 *   backward  g[i, v] = dloss[i] * (exp(z[i, v] - lse[i]) - [v == t[i]]),
 *             dhidden = g @ weight,  dweight = g^T @ hidden.
 * A negative target marks an ignored row: loss 0, no gradient.
 *
 * Layouts (row-major, DEVICE pointers, 16-byte aligned, owned by the caller):
 *   hidden  [N, Dm]   weight [V, Dm]   (dtype: bf16 or fp16, the same for both)
 *   targets [N] int32 (-1 or any negative = ignored; else < V)
 *   loss, lse, dloss [N] float32 (lse in natural log)
 *   dhidden [N, Dm], dweight [V, Dm] in the input dtype, fully overwritten.
 * Shapes: N, Dm, V >= 1 and Dm a multiple of 64 (else ATTN_ERR_UNSUPPORTED).
 *
 * workspace: DEVICE pointer, 16-byte aligned, at least lce_workspace_bytes(N,
 *   Dm, V) bytes (0 means the shape is rejected); contents on entry ignored,
 *   undefined on exit; not shared by two calls in flight.  The forward keeps
 *   one (max, sum) pair per row and 256-entry vocabulary tile there; the
 *   backward keeps one chunk of g (16384 vocabulary entries, 16-bit) and an
 *   fp32 dhidden accumulator.
 * Products: every product runs in this library's tcgen05 kernels: the
 *   logits tiles with their epilogues, and the backward's two products per
 *   vocabulary chunk (dhidden += g W_chunk with an fp32 sum across chunks,
 *   rounded to 16 bits once at the end; dweight_chunk = g^T hidden, fp32
 *   accumulation, rounded to 16 bits).  No other library is called.
 * Errors: a null or misaligned pointer, N, Dm or V < 1, a bad dtype or a small
 *   workspace is ATTN_ERR_INVALID_ARG; Dm % 64 != 0 is ATTN_ERR_UNSUPPORTED;
 *   a failed launch is ATTN_ERR_CUDA.  A target >= V is treated like a
 *   negative one (ignored row).
 */
#ifndef GBLCE_H_
#define GBLCE_H_

#include <stddef.h>
#include <stdint.h>

#include "gbattn.h"

#ifdef __cplusplus
extern "C" {
#endif

size_t lce_workspace_bytes(int N, int Dm, int V);

attn_status_t lce_fwd(const void* hidden, const void* weight, const int32_t* targets, float* loss, float* lse,
                      void* workspace, size_t workspace_bytes, int N, int Dm, int V, attn_dtype_t dtype,
                      cudaStream_t stream);

attn_status_t lce_bwd(const void* hidden, const void* weight, const int32_t* targets, const float* lse,
                      const float* dloss, void* dhidden, void* dweight, void* workspace, size_t workspace_bytes,
                      int N, int Dm, int V, attn_dtype_t dtype, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* GBLCE_H_ */
