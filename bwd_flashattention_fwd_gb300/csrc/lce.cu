// C ABI of the linear cross-entropy calls (declared in include/gblce.h):
// validation, tensor maps, the logits-tile kernels of lce_kernel.cuh and, in
// the backward, the two gradient products of lce_gemm_kernel.cuh per
// vocabulary chunk.
#include "../../include/gblce.h"
#include "launch.h"
#include "lce_gemm_kernel.cuh"
#include "lce_kernel.cuh"

namespace gbattn {
namespace {

constexpr int kLceVocabChunk = 16384;  // vocabulary entries per backward chunk (64 tiles)

size_t round16(size_t x) { return (x + 15) & ~static_cast<size_t>(15); }

int vocab_tiles(int v) { return (v + LceGeom::BN - 1) / LceGeom::BN; }

// Columns of the backward's g chunk (a whole number of tiles).
int chunk_cols(int V) {
  const int full = vocab_tiles(V) * LceGeom::BN;
  return full < kLceVocabChunk ? full : kLceVocabChunk;
}

size_t ws_forward(int N, int V) {
  return round16(static_cast<size_t>(vocab_tiles(V)) * N * sizeof(float2)) + round16(static_cast<size_t>(N) * 4);
}

size_t ws_backward(int N, int Dm, int V) {
  return round16(static_cast<size_t>(N) * chunk_cols(V) * 2) + static_cast<size_t>(N) * Dm * 4;
}

attn_status_t check_lce(int N, int Dm, int V, attn_dtype_t dtype) {
  if (N < 1 || Dm < 1 || V < 1) return ATTN_ERR_INVALID_ARG;
  if (dtype != ATTN_DTYPE_FP16 && dtype != ATTN_DTYPE_BF16) return ATTN_ERR_INVALID_ARG;
  if (Dm % LceGeom::BK != 0) return ATTN_ERR_UNSUPPORTED;
  // tile counts and GEMM sizes are ints
  if (static_cast<long long>(vocab_tiles(V)) * ((N + LceGeom::BM - 1) / LceGeom::BM) > 0x7fffffffLL)
    return ATTN_ERR_UNSUPPORTED;
  return ATTN_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Rank-3 view [1, rows, Dm] of a row-major [rows, Dm] matrix, 64-column x
// box_rows boxes with the 128-byte swizzle; rows past `rows` read as zeros.
bool lce_map(EncodeTiledFn enc, CUtensorMap* m, const void* base, int rows, int Dm, int box_rows, bool bf16) {
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(Dm), static_cast<cuuint64_t>(rows), 1};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(Dm) * 2,
                                 static_cast<cuuint64_t>(Dm) * 2 * static_cast<cuuint64_t>(rows)};
  const cuuint32_t box[3] = {64u, static_cast<cuuint32_t>(box_rows), 1u};
  const cuuint32_t elem_strides[3] = {1u, 1u, 1u};
  return enc(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void*>(base),
             dims, strides, box, elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <bool BF16, bool GRAD>
int launch_logits(const LceParams& p, const CUtensorMap& tmH, const CUtensorMap& tmW, int num_sms,
                  cudaStream_t stream) {
  auto kern = lce_logits_kernel<BF16, GRAD>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, LceGeom::SMEM_BYTES) != cudaSuccess)
    return kLaunchCudaError;
  const long long tiles = static_cast<long long>(p.n_vt) * p.n_rt;
  const int grid = static_cast<int>(tiles < num_sms ? tiles : num_sms);
  kern<<<grid, LceGeom::NUM_THREADS, LceGeom::SMEM_BYTES, stream>>>(tmH, tmW, p);
  return cudaPeekAtLastError() == cudaSuccess ? kLaunchOk : kLaunchCudaError;
}

template <bool BF16, bool A_MN>
int launch_gemm(const LceGemmParams& p, const CUtensorMap& tmA, const CUtensorMap& tmB, int num_sms,
                cudaStream_t stream) {
  auto kern = lce_gemm_kernel<BF16, A_MN>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, LceGemmGeom::SMEM_BYTES) !=
      cudaSuccess)
    return kLaunchCudaError;
  const long long tiles = static_cast<long long>(p.n_mt) * p.n_nt;
  const int grid = static_cast<int>(tiles < num_sms ? tiles : num_sms);
  kern<<<grid, LceGemmGeom::NUM_THREADS, LceGemmGeom::SMEM_BYTES, stream>>>(tmA, tmB, p);
  return cudaPeekAtLastError() == cudaSuccess ? kLaunchOk : kLaunchCudaError;
}

template <bool BF16>
int launch_gemm_pair(const LceGemmParams& dh, const CUtensorMap& tmGk, const CUtensorMap& tmWn,
                     const LceGemmParams& dw, const CUtensorMap& tmGm, const CUtensorMap& tmHn, int num_sms,
                     cudaStream_t stream) {
  const int r = launch_gemm<BF16, false>(dh, tmGk, tmWn, num_sms, stream);
  return r != kLaunchOk ? r : launch_gemm<BF16, true>(dw, tmGm, tmHn, num_sms, stream);
}

attn_status_t finish(int r) {
  if (r == kLaunchOk) return ATTN_OK;
  if (r == kLaunchBadMap) return ATTN_ERR_INVALID_ARG;
  return ATTN_ERR_CUDA;
}

}  // namespace
}  // namespace gbattn

using namespace gbattn;

extern "C" size_t lce_workspace_bytes(int N, int Dm, int V) {
  if (check_lce(N, Dm, V, ATTN_DTYPE_BF16) != ATTN_OK) return 0;
  const size_t f = ws_forward(N, V), b = ws_backward(N, Dm, V);
  return f > b ? f : b;
}

extern "C" attn_status_t lce_fwd(const void* hidden, const void* weight, const int32_t* targets, float* loss,
                                 float* lse, void* workspace, size_t workspace_bytes, int N, int Dm, int V,
                                 attn_dtype_t dtype, cudaStream_t stream) {
  if (!hidden || !weight || !targets || !loss || !lse || !workspace) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(hidden) || !aligned16(weight) || !aligned16(targets) || !aligned16(loss) || !aligned16(lse) ||
      !aligned16(workspace))
    return ATTN_ERR_INVALID_ARG;
  const attn_status_t s = check_lce(N, Dm, V, dtype);
  if (s != ATTN_OK) return s;
  if (workspace_bytes < ws_forward(N, V)) return ATTN_ERR_INVALID_ARG;
  int dev, num_sms, *status;
  EncodeTiledFn enc;
  const attn_status_t ds = shared_device_state(&dev, &enc, &status, &num_sms);
  if (ds != ATTN_OK) return ds;
  const bool bf16 = dtype == ATTN_DTYPE_BF16;
  CUtensorMap tmH, tmW;
  if (!lce_map(enc, &tmH, hidden, N, Dm, LceGeom::BM, bf16) || !lce_map(enc, &tmW, weight, V, Dm, LceGeom::BN, bf16))
    return ATTN_ERR_INVALID_ARG;
  LceParams p{};
  p.N = N, p.Dm = Dm, p.V = V;
  p.n_rt = (N + LceGeom::BM - 1) / LceGeom::BM;
  p.n_vt = vocab_tiles(V);
  p.v0 = 0, p.v_end = V;
  p.targets = targets;
  p.part = static_cast<float2*>(workspace);
  p.tgt_logit = reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                         round16(static_cast<size_t>(p.n_vt) * N * sizeof(float2)));
  p.status = status;
  p.limit_ns = shared_wait_limit_ns();
  const int r = bf16 ? launch_logits<true, false>(p, tmH, tmW, num_sms, stream)
                     : launch_logits<false, false>(p, tmH, tmW, num_sms, stream);
  if (r != kLaunchOk) return finish(r);
  lce_combine_kernel<<<(N + 255) / 256, 256, 0, stream>>>(p.part, p.tgt_logit, targets, p.n_vt, N, V, loss,
                                                            lse);
  return cudaPeekAtLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

extern "C" attn_status_t lce_bwd(const void* hidden, const void* weight, const int32_t* targets, const float* lse,
                                 const float* dloss, void* dhidden, void* dweight, void* workspace,
                                 size_t workspace_bytes, int N, int Dm, int V, attn_dtype_t dtype,
                                 cudaStream_t stream) {
  if (!hidden || !weight || !targets || !lse || !dloss || !dhidden || !dweight || !workspace)
    return ATTN_ERR_INVALID_ARG;
  if (!aligned16(hidden) || !aligned16(weight) || !aligned16(targets) || !aligned16(lse) || !aligned16(dloss) ||
      !aligned16(dhidden) || !aligned16(dweight) || !aligned16(workspace))
    return ATTN_ERR_INVALID_ARG;
  const attn_status_t s = check_lce(N, Dm, V, dtype);
  if (s != ATTN_OK) return s;
  if (workspace_bytes < ws_backward(N, Dm, V)) return ATTN_ERR_INVALID_ARG;
  int dev, num_sms, *status;
  EncodeTiledFn enc;
  const attn_status_t ds = shared_device_state(&dev, &enc, &status, &num_sms);
  if (ds != ATTN_OK) return ds;
  const bool bf16 = dtype == ATTN_DTYPE_BF16;
  const int ldg = chunk_cols(V);
  void* g = workspace;
  float* dh32 = reinterpret_cast<float*>(static_cast<char*>(workspace) + round16(static_cast<size_t>(N) * ldg * 2));
  // logits tiles (K-major H and W); the products: g K-major [N][ldg] for dH,
  // g MN-major (read transposed) for dW, W and H MN-major
  CUtensorMap tmH, tmW, tmGk, tmGm, tmWn, tmHn;
  if (!lce_map(enc, &tmH, hidden, N, Dm, LceGeom::BM, bf16) || !lce_map(enc, &tmW, weight, V, Dm, LceGeom::BN, bf16) ||
      !lce_map(enc, &tmGk, g, N, ldg, LceGemmGeom::BM, bf16) || !lce_map(enc, &tmGm, g, N, ldg, 64, bf16) ||
      !lce_map(enc, &tmWn, weight, V, Dm, 64, bf16) || !lce_map(enc, &tmHn, hidden, N, Dm, 64, bf16))
    return ATTN_ERR_INVALID_ARG;
  LceParams p{};
  p.N = N, p.Dm = Dm, p.V = V;
  p.n_rt = (N + LceGeom::BM - 1) / LceGeom::BM;
  p.targets = targets;
  p.lse = lse, p.dloss = dloss, p.g = g, p.ldg = ldg;
  p.status = status;
  p.limit_ns = shared_wait_limit_ns();
  const int n_ht = (Dm + LceGemmGeom::BN - 1) / LceGemmGeom::BN;  // tiles along the hidden size
  for (int v0 = 0; v0 < V; v0 += ldg) {
    const int vc = V - v0 < ldg ? V - v0 : ldg;
    const bool first = v0 == 0, last = v0 + vc >= V;
    p.v0 = v0, p.v_end = v0 + vc, p.n_vt = vocab_tiles(vc);
    int r = bf16 ? launch_logits<true, true>(p, tmH, tmW, num_sms, stream)
                 : launch_logits<false, true>(p, tmH, tmW, num_sms, stream);
    if (r != kLaunchOk) return finish(r);
    // dhidden (+)= g [N, vc] W[v0 : v0 + vc]: fp32 sum over the chunks in the
    // workspace, rounded to 16 bits into dhidden by the last chunk
    LceGemmParams dh{};
    dh.M = N, dh.N = Dm, dh.n_mt = p.n_rt, dh.n_nt = n_ht, dh.n_kt = (vc + LceGemmGeom::BK - 1) / LceGemmGeom::BK;
    dh.b_k0 = v0;
    dh.acc_in = first ? nullptr : dh32;
    dh.acc_out = last ? nullptr : dh32;
    dh.out16 = last ? dhidden : nullptr;
    dh.ldc = Dm, dh.status = status, dh.limit_ns = p.limit_ns;
    // dweight[v0 : v0 + vc] = g^T hidden
    LceGemmParams dw{};
    dw.M = vc, dw.N = Dm, dw.n_mt = (vc + LceGemmGeom::BM - 1) / LceGemmGeom::BM, dw.n_nt = n_ht;
    dw.n_kt = (N + LceGemmGeom::BK - 1) / LceGemmGeom::BK;
    dw.b_k0 = 0;
    dw.out16 = static_cast<char*>(dweight) + static_cast<size_t>(v0) * Dm * 2;
    dw.ldc = Dm, dw.status = status, dw.limit_ns = p.limit_ns;
    r = bf16 ? launch_gemm_pair<true>(dh, tmGk, tmWn, dw, tmGm, tmHn, num_sms, stream)
             : launch_gemm_pair<false>(dh, tmGk, tmWn, dw, tmGm, tmHn, num_sms, stream);
    if (r != kLaunchOk) return finish(r);
  }
  return ATTN_OK;
}
