// Kernel instantiations and launchers for one head dimension.  The build
// compiles this file once per supported D with -DGBATTN_HEAD_DIM=<D>, so the
// four translation units compile in parallel.
#include "launch.h"

#include "bwd_dkv2_kernel.cuh"
#include "bwd_dkv_kernel.cuh"
#include "bwd_dq3_kernel.cuh"
#include "bwd_dq_kernel.cuh"
#include "decode_kernel.cuh"
#include "delta_kernel.cuh"
#include "fwd2_kernel.cuh"
#include "fwd_kernel.cuh"

#ifndef GBATTN_HEAD_DIM
#error "compile with -DGBATTN_HEAD_DIM=<64|96|128|256>"
#endif

#define GBATTN_CAT2(a, b) a##b
#define GBATTN_CAT(a, b) GBATTN_CAT2(a, b)

namespace gbattn {
// A namespace per head dimension: the four objects are built from this one
// file and are linked together.
namespace GBATTN_CAT(inst_d, GBATTN_HEAD_DIM) {

constexpr int kD = GBATTN_HEAD_DIM;

// Rank-3 view [B*H, L, D] of a [B, H, pitch, D] tensor (contiguous when
// pitch = L; a slice of the first L rows of each head otherwise); boxes of
// 64 columns x box_rows rows with the 128-byte swizzle the MMA descriptors
// expect.  Rows past L (and columns past D) read as zeros, so rows behind a
// slice are never read.
bool make_map(const AttnArgs& a, CUtensorMap* m, const void* base, int L, int BH, int box_rows,
              int64_t pitch = 0) {
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(L),
                              static_cast<cuuint64_t>(BH)};
  const cuuint64_t rows = static_cast<cuuint64_t>(pitch > 0 ? pitch : L);
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(kD) * 2, static_cast<cuuint64_t>(kD) * 2 * rows};
  const cuuint32_t box[3] = {64u, static_cast<cuuint32_t>(box_rows), 1u};
  const cuuint32_t elem_strides[3] = {1u, 1u, 1u};
  const CUresult r = a.encode(m, a.bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                              3, const_cast<void*>(base), dims, strides, box, elem_strides,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <typename Kern>
int launch(Kern kern, dim3 grid, int threads, int smem, cudaStream_t stream, const CUtensorMap& a0,
           const CUtensorMap& a1, const CUtensorMap& a2, const FwdParams& p) {
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return kLaunchCudaError;
  kern<<<grid, threads, smem, stream>>>(a0, a1, a2, p);
  return cudaPeekAtLastError() == cudaSuccess ? kLaunchOk : kLaunchCudaError;
}

template <typename Kern>
int launch(Kern kern, dim3 grid, int threads, int smem, cudaStream_t stream, const CUtensorMap& a0,
           const CUtensorMap& a1, const CUtensorMap& a2, const CUtensorMap& a3, const BwdParams& p) {
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return kLaunchCudaError;
  kern<<<grid, threads, smem, stream>>>(a0, a1, a2, a3, p);
  return cudaPeekAtLastError() == cudaSuccess ? kLaunchOk : kLaunchCudaError;
}

// Launch as a programmatic dependent of the previous kernel on the stream:
// its CTAs may start while that kernel finishes, so the kernel waits for it
// (griddepcontrol.wait) before reading anything in global memory.
template <typename Kern, typename... Args>
int launch_dependent(Kern kern, dim3 grid, int threads, int smem, cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kern, args...) != cudaSuccess) return kLaunchCudaError;
  return cudaPeekAtLastError() == cudaSuccess ? kLaunchOk : kLaunchCudaError;
}

// D <= 128: two 128-row query tiles per work item, persistent CTAs (fwd2_kernel.cuh).
template <bool BF16, bool CAUSAL, bool MASKED>
int fwd2_impl(const AttnArgs& a) {
  using Gm = Fwd2Geom<(kD <= 128 ? kD : 128)>;
  CUtensorMap tq, tk, tv, to;
  // O is written by TMA stores of one softmax warp's 32 rows
  if (!make_map(a, &tq, a.q, a.Lq, a.B * a.Hq, Gm::BQ) ||
      !make_map(a, &tk, a.k, a.Lk, a.B * a.Hkv, Gm::BK, a.kv_pitch) ||
      !make_map(a, &tv, a.v, a.Lk, a.B * a.Hkv, Gm::BK, a.kv_pitch) ||
      !make_map(a, &to, a.o_out, a.Lq, a.B * a.Hq, 32))
    return kLaunchBadMap;
  FwdParams p{};
  p.o = a.o_out;
  p.lse = a.lse_out;
  p.status = a.status;
  p.B = a.B, p.Hq = a.Hq, p.Hkv = a.Hkv, p.Lq = a.Lq, p.Lk = a.Lk, p.G = a.Hq / a.Hkv;
  p.off = a.Lk - a.Lq;
  p.n_qtiles = (a.Lq + 2 * Gm::BQ - 1) / (2 * Gm::BQ);  // 256-row pairs of tiles
  p.bmask = a.block_mask;
  p.nkb = (a.Lk + kMaskBlock - 1) / kMaskBlock;
  p.scale_log2 = static_cast<float>(static_cast<double>(a.scale) * 1.4426950408889634074);
  p.limit_ns = a.limit_ns;
  p.sched = a.sched;
  // persistent: one CTA per SM (fewer when there are fewer work items)
  const long long n_items = static_cast<long long>(p.n_qtiles) * a.B * a.Hq;
  const int sms = a.num_sms > 0 ? a.num_sms : 1;
  const dim3 grid(static_cast<unsigned>(n_items < sms ? n_items : sms));
  auto kern = attn_fwd2_kernel<(kD <= 128 ? kD : 128), BF16, CAUSAL, MASKED>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Gm::SMEM_BYTES) != cudaSuccess)
    return kLaunchCudaError;
  kern<<<grid, Gm::NUM_THREADS, Gm::SMEM_BYTES, a.stream>>>(tq, tk, tv, to, p);
  return cudaPeekAtLastError() == cudaSuccess ? kLaunchOk : kLaunchCudaError;
}

template <bool BF16, bool CAUSAL>
int fwd_impl(const AttnArgs& a) {
  if constexpr (kD <= 128) {
    return a.block_mask ? fwd2_impl<BF16, CAUSAL, true>(a) : fwd2_impl<BF16, CAUSAL, false>(a);
  } else {
    using Gm = FwdGeom<kD>;
    CUtensorMap tq, tk, tv;
    if (!make_map(a, &tq, a.q, a.Lq, a.B * a.Hq, Gm::BQ) ||
        !make_map(a, &tk, a.k, a.Lk, a.B * a.Hkv, Gm::BK, a.kv_pitch) ||
        !make_map(a, &tv, a.v, a.Lk, a.B * a.Hkv, Gm::BK, a.kv_pitch))
      return kLaunchBadMap;
    FwdParams p{};
    p.o = a.o_out;
    p.lse = a.lse_out;
    p.status = a.status;
    p.B = a.B, p.Hq = a.Hq, p.Hkv = a.Hkv, p.Lq = a.Lq, p.Lk = a.Lk, p.G = a.Hq / a.Hkv;
    p.off = a.Lk - a.Lq;
    p.n_qtiles = (a.Lq + Gm::BQ - 1) / Gm::BQ;
    p.scale_log2 = static_cast<float>(static_cast<double>(a.scale) * 1.4426950408889634074);
    p.limit_ns = a.limit_ns;
    p.bmask = a.block_mask;
    p.nkb = (a.Lk + kMaskBlock - 1) / kMaskBlock;
    const dim3 grid(a.B * a.Hq, p.n_qtiles);
    if (a.block_mask)
      return launch(attn_fwd_kernel<kD, BF16, CAUSAL, false, true>, grid, Gm::NUM_THREADS, Gm::SMEM_BYTES, a.stream,
                    tq, tk, tv, p);
    return launch(attn_fwd_kernel<kD, BF16, CAUSAL>, grid, Gm::NUM_THREADS, Gm::SMEM_BYTES, a.stream, tq, tk,
                  tv, p);
  }
}

BwdParams bwd_params(const AttnArgs& a) {
  BwdParams p{};
  p.dq = a.dq;
  p.dk = a.dk;
  p.dv = a.dv;
  p.lse = a.lse;
  p.delta = a.delta;
  p.status = a.status;
  p.B = a.B, p.Hq = a.Hq, p.Hkv = a.Hkv, p.Lq = a.Lq, p.Lk = a.Lk, p.G = a.Hq / a.Hkv;
  p.off = a.Lk - a.Lq;
  p.scale = a.scale;
  p.scale_log2 = static_cast<float>(static_cast<double>(a.scale) * 1.4426950408889634074);
  p.limit_ns = a.limit_ns;
  p.bmask = a.block_mask;
  p.nkb = (a.Lk + kMaskBlock - 1) / kMaskBlock;
  p.kv_pitch = a.kv_pitch > 0 ? a.kv_pitch : a.Lk;
  p.k = a.k;
  p.v = a.v;
  return p;
}

// D = 256: the dV and dK halves in one launch (bwd_dkv_kernel.cuh).  A
// template of its own so that only the D = 256 unit instantiates the kernel.
template <int DD, bool BF16, bool CAUSAL>
int dkv256_impl(const AttnArgs& a) {
  static_assert(DD == 256, "the pair kernel is the D = 256 dK/dV path");
  using Gm = DkvPairGeom;
  CUtensorMap tq, tdo;
  if (!make_map(a, &tq, a.q, a.Lq, a.B * a.Hq, Gm::BQ) || !make_map(a, &tdo, a.dO, a.Lq, a.B * a.Hq, Gm::BQ))
    return kLaunchBadMap;
  BwdParams p = bwd_params(a);
  p.n_qtiles = (a.Lq + Gm::BQ - 1) / Gm::BQ;
  p.n_ktiles = (a.Lk + Gm::BK - 1) / Gm::BK;
  const dim3 grid(2 * a.B * a.Hkv, p.n_ktiles);  // x: the two CTAs of a cluster
  auto kern = a.block_mask ? attn_bwd_dkv_kernel<BF16, CAUSAL, true> : attn_bwd_dkv_kernel<BF16, CAUSAL, false>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Gm::SMEM_BYTES) != cudaSuccess)
    return kLaunchCudaError;
  kern<<<grid, Gm::NUM_THREADS, Gm::SMEM_BYTES, a.stream>>>(tq, tdo, p);
  return cudaPeekAtLastError() == cudaSuccess ? kLaunchOk : kLaunchCudaError;
}

// D <= 128: K held in tensor memory as the A operand of S^T (bwd_dkv2_kernel.cuh).
template <bool BF16, bool CAUSAL, bool MASKED>
int dkv2_impl(const AttnArgs& a) {
  constexpr int DD = kD <= 128 ? kD : 128;
  using Gm = Dkv2Geom<DD>;
  CUtensorMap tq, tv, tdo;
  if (!make_map(a, &tq, a.q, a.Lq, a.B * a.Hq, Gm::BQ) || !make_map(a, &tdo, a.dO, a.Lq, a.B * a.Hq, Gm::BQ) ||
      !make_map(a, &tv, a.v, a.Lk, a.B * a.Hkv, Gm::BK, a.kv_pitch))
    return kLaunchBadMap;
  BwdParams p = bwd_params(a);
  p.n_qtiles = (a.Lq + Gm::BQ - 1) / Gm::BQ;
  p.n_ktiles = (a.Lk + Gm::BK - 1) / Gm::BK;
  const dim3 grid(a.B * a.Hkv, p.n_ktiles);
  auto kern = attn_bwd_dkv2_kernel<DD, BF16, CAUSAL, MASKED>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Gm::SMEM_BYTES) != cudaSuccess)
    return kLaunchCudaError;
  // behind the delta kernel: its CTAs start as that kernel's retire
  return launch_dependent(kern, grid, Gm::NUM_THREADS, Gm::SMEM_BYTES, a.stream, tq, tv, tdo, a.k, p);
}

// D <= 128: Q and dO held in tensor memory as MMA A operands (bwd_dq3_kernel.cuh).
// behind_dkv: launched right behind the dK/dV kernel on the same stream as a
// programmatic dependent, so its CTAs fill the SMs the dK/dV kernel's last
// wave frees (it reads none of that kernel's outputs).
template <bool BF16, bool CAUSAL, bool MASKED>
int dq3_impl(const AttnArgs& a, bool behind_dkv) {
  constexpr int DD = kD <= 128 ? kD : 128;
  using Gm = Dq3Geom<DD>;
  CUtensorMap tq, tdo, tk, tv, tdq;
  // dQ is written by TMA stores of 32-row tiles
  if (!make_map(a, &tq, a.q, a.Lq, a.B * a.Hq, Gm::BQ) || !make_map(a, &tdo, a.dO, a.Lq, a.B * a.Hq, Gm::BQ) ||
      !make_map(a, &tk, a.k, a.Lk, a.B * a.Hkv, Gm::BK, a.kv_pitch) ||
      !make_map(a, &tv, a.v, a.Lk, a.B * a.Hkv, Gm::BK, a.kv_pitch) ||
      !make_map(a, &tdq, a.dq, a.Lq, a.B * a.Hq, 32))
    return kLaunchBadMap;
  BwdParams p = bwd_params(a);
  p.n_qtiles = (a.Lq + Gm::BQ - 1) / Gm::BQ;
  p.n_ktiles = (a.Lk + Gm::BK - 1) / Gm::BK;
  // persistent: one CTA per SM (fewer when there are fewer work items)
  const long long n_items = static_cast<long long>(p.n_qtiles) * a.B * a.Hq;
  const int sms = a.num_sms > 0 ? a.num_sms : 1;
  const dim3 grid(static_cast<unsigned>(n_items < sms ? n_items : sms));
  p.sched = a.sched;
  auto kern = attn_bwd_dq3_kernel<DD, BF16, CAUSAL, MASKED>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Gm::SMEM_BYTES) != cudaSuccess)
    return kLaunchCudaError;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(Gm::NUM_THREADS);
  cfg.dynamicSmemBytes = Gm::SMEM_BYTES;
  cfg.stream = a.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = behind_dkv ? 1 : 0;
  if (cudaLaunchKernelEx(&cfg, kern, tq, tdo, tk, tv, tdq, p) != cudaSuccess) return kLaunchCudaError;
  return cudaPeekAtLastError() == cudaSuccess ? kLaunchOk : kLaunchCudaError;
}

template <bool BF16, bool CAUSAL>
int dq_impl(const AttnArgs& a, bool behind_dkv = false) {
  if constexpr (kD <= 128) {
    return a.block_mask ? dq3_impl<BF16, CAUSAL, true>(a, behind_dkv) : dq3_impl<BF16, CAUSAL, false>(a, behind_dkv);
  } else {
    using Gm = DqGeom<kD>;
    CUtensorMap tq, tk, tv, tdo;
    if (!make_map(a, &tq, a.q, a.Lq, a.B * a.Hq, Gm::BQ) || !make_map(a, &tdo, a.dO, a.Lq, a.B * a.Hq, Gm::BQ) ||
        !make_map(a, &tk, a.k, a.Lk, a.B * a.Hkv, Gm::BK, a.kv_pitch) ||
        !make_map(a, &tv, a.v, a.Lk, a.B * a.Hkv, Gm::BK, a.kv_pitch))
      return kLaunchBadMap;
    BwdParams p = bwd_params(a);
    p.n_qtiles = (a.Lq + Gm::BQ - 1) / Gm::BQ;
    p.n_ktiles = (a.Lk + Gm::BK - 1) / Gm::BK;
    const dim3 grid(a.B * a.Hq, p.n_qtiles);
    auto kern = a.block_mask ? attn_bwd_dq_kernel<kD, BF16, CAUSAL, false, true> : attn_bwd_dq_kernel<kD, BF16, CAUSAL>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Gm::SMEM_BYTES) != cudaSuccess)
      return kLaunchCudaError;
    // behind the dK/dV kernel: the hardware hands this grid's CTAs to the
    // SMs that kernel's last wave frees (its CTAs run in any order anyway)
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(Gm::NUM_THREADS);
    cfg.dynamicSmemBytes = Gm::SMEM_BYTES;
    cfg.stream = a.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = behind_dkv ? 1 : 0;
    if (cudaLaunchKernelEx(&cfg, kern, tq, tk, tv, tdo, p) != cudaSuccess) return kLaunchCudaError;
    return cudaPeekAtLastError() == cudaSuccess ? kLaunchOk : kLaunchCudaError;
  }
}

template <bool BF16, bool CAUSAL>
int dkv_all(const AttnArgs& a) {
  if constexpr (kD <= 128) {
    return a.block_mask ? dkv2_impl<BF16, CAUSAL, true>(a) : dkv2_impl<BF16, CAUSAL, false>(a);
  } else {
    return dkv256_impl<kD, BF16, CAUSAL>(a);
  }
}

template <bool BF16, bool CAUSAL>
int bwd_impl(const AttnArgs& a) {
  const int r = dkv_all<BF16, CAUSAL>(a);
  return r == kLaunchOk ? dq_impl<BF16, CAUSAL>(a, /*behind_dkv=*/true) : r;
}

// Decode-shaped forward (G * Lq <= 128): the single-tile forward kernel on
// packed tiles, its key range split over CTAs, then the combine kernel.
template <bool BF16, bool CAUSAL>
int fwd_decode_impl(const AttnArgs& a) {
  using Gm = FwdGeom<kD>;
  const int R = (a.Hq / a.Hkv) * a.Lq;  // packed rows of one KV head
  const long long groups = static_cast<long long>(a.B) * a.Hkv;
  const long long nrows = groups * R;
  CUtensorMap tq, tk, tv;
  if (!make_map(a, &tq, a.q, R, a.B * a.Hkv, Gm::BQ) ||
      !make_map(a, &tk, a.k, a.Lk, a.B * a.Hkv, Gm::BK, a.kv_pitch) ||
      !make_map(a, &tv, a.v, a.Lk, a.B * a.Hkv, Gm::BK, a.kv_pitch))
    return kLaunchBadMap;
  const DecodeSplit sp = decode_split(groups, decode_fwd_tiles(a.Lk, kD));
  FwdParams p{};
  p.status = a.status;
  p.B = a.B, p.Hq = a.Hkv, p.Hkv = a.Hkv, p.Lq = R, p.Lk = a.Lk, p.G = 1;
  p.off = a.Lk - a.Lq;  // from the true query length
  p.n_qtiles = 1;
  p.scale_log2 = static_cast<float>(static_cast<double>(a.scale) * 1.4426950408889634074);
  p.limit_ns = a.limit_ns;
  p.qmod = a.Lq;
  p.split_tiles = sp.tiles_per_split;
  p.ws = a.workspace;
  p.ws_lse = a.workspace + static_cast<size_t>(sp.n_split) * nrows * kD;
  const dim3 grid(static_cast<unsigned>(groups), sp.n_split);
  const int r = launch(attn_fwd_kernel<kD, BF16, CAUSAL, true>, grid, Gm::NUM_THREADS, Gm::SMEM_BYTES, a.stream, tq,
                       tk, tv, p);
  if (r != kLaunchOk) return r;
  const long long blocks = (nrows + kCombineThreads / 32 - 1) / (kCombineThreads / 32);
  attn_decode_combine_kernel<kD, BF16><<<static_cast<unsigned>(blocks), kCombineThreads, 0, a.stream>>>(
      p.ws, p.ws_lse, sp.n_split, nrows, a.o_out, a.lse_out);
  return cudaPeekAtLastError() == cudaSuccess ? kLaunchOk : kLaunchCudaError;
}

// Decode-shaped dQ: the single-tile dQ kernel on packed tiles, its key range
// split over CTAs, then the reduction of the fp32 shares.
template <bool BF16, bool CAUSAL>
int dq_decode_impl(const AttnArgs& a) {
  using Gm = DqGeom<kD>;
  const int R = (a.Hq / a.Hkv) * a.Lq;
  const long long groups = static_cast<long long>(a.B) * a.Hkv;
  const long long nrows = groups * R;
  CUtensorMap tq, tk, tv, tdo;
  if (!make_map(a, &tq, a.q, R, a.B * a.Hkv, Gm::BQ) || !make_map(a, &tdo, a.dO, R, a.B * a.Hkv, Gm::BQ) ||
      !make_map(a, &tk, a.k, a.Lk, a.B * a.Hkv, Gm::BK, a.kv_pitch) ||
      !make_map(a, &tv, a.v, a.Lk, a.B * a.Hkv, Gm::BK, a.kv_pitch))
    return kLaunchBadMap;
  const DecodeSplit sp = decode_split(groups, decode_dq_tiles(a.Lk));
  BwdParams p = bwd_params(a);  // off = Lk - Lq from the true query length
  p.Hq = a.Hkv, p.Lq = R, p.G = 1;
  p.n_qtiles = 1;
  p.n_ktiles = decode_dq_tiles(a.Lk);
  p.qmod = a.Lq;
  p.split_tiles = sp.tiles_per_split;
  p.ws = a.workspace;
  const dim3 grid(static_cast<unsigned>(groups), sp.n_split);
  auto kern = attn_bwd_dq_kernel<kD, BF16, CAUSAL, true>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Gm::SMEM_BYTES) != cudaSuccess)
    return kLaunchCudaError;
  // behind the decode dK/dV kernel: its CTAs take the SMs that kernel frees
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(Gm::NUM_THREADS);
  cfg.dynamicSmemBytes = Gm::SMEM_BYTES;
  cfg.stream = a.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = a.dq_behind_dkv ? 1 : 0;
  const int r = cudaLaunchKernelEx(&cfg, kern, tq, tk, tv, tdo, p) == cudaSuccess ? kLaunchOk : kLaunchCudaError;
  if (r != kLaunchOk) return r;
  const long long n4 = nrows * kD / 4;
  long long blocks = (n4 + kReduceThreads - 1) / kReduceThreads;
  const long long cap = static_cast<long long>(a.num_sms > 0 ? a.num_sms : 152) * 8;
  if (blocks > cap) blocks = cap;
  attn_decode_dq_reduce_kernel<kD, BF16><<<static_cast<unsigned>(blocks), kReduceThreads, 0, a.stream>>>(
      p.ws, sp.n_split, nrows, a.scale, a.dq);
  return cudaPeekAtLastError() == cudaSuccess ? kLaunchOk : kLaunchCudaError;
}

// Decode-shaped dK/dV: D <= 128 streams each KV head's key tiles against its
// one packed query tile (decode_kernel.cuh); D = 256 runs the general pair.
template <bool BF16, bool CAUSAL>
int dkv_decode_impl(const AttnArgs& a) {
  if constexpr (kD <= 128) {
    constexpr int DD = kD <= 128 ? kD : 128;  // (this branch is compiled for every D)
    using Gm = DecodeDkvGeom<DD>;
    const int R = (a.Hq / a.Hkv) * a.Lq;
    const long long groups = static_cast<long long>(a.B) * a.Hkv;
    CUtensorMap tq, tk, tv, tdo;
    if (!make_map(a, &tq, a.q, R, a.B * a.Hkv, Gm::RQ) || !make_map(a, &tdo, a.dO, R, a.B * a.Hkv, Gm::RQ) ||
        !make_map(a, &tk, a.k, a.Lk, a.B * a.Hkv, Gm::BK, a.kv_pitch) ||
        !make_map(a, &tv, a.v, a.Lk, a.B * a.Hkv, Gm::BK, a.kv_pitch))
      return kLaunchBadMap;
    BwdParams p = bwd_params(a);  // off = Lk - Lq from the true query length
    p.Hq = a.Hkv, p.Lq = R, p.G = 1;
    p.qmod = a.Lq;
    p.n_ktiles = (a.Lk + Gm::BK - 1) / Gm::BK;
    const DecodeSplit sp = decode_split(groups, p.n_ktiles);
    p.split_tiles = sp.tiles_per_split;
    const dim3 grid(static_cast<unsigned>(groups), sp.n_split);
    auto kern = attn_decode_dkv_kernel<DD, BF16, CAUSAL>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Gm::SMEM_BYTES) != cudaSuccess)
      return kLaunchCudaError;
    kern<<<grid, Gm::NUM_THREADS, Gm::SMEM_BYTES, a.stream>>>(tq, tk, tv, tdo, p);
    return cudaPeekAtLastError() == cudaSuccess ? kLaunchOk : kLaunchCudaError;
  } else {
    return dkv_all<BF16, CAUSAL>(a);
  }
}

template <bool BF16>
int delta_impl(const AttnArgs& a) {
  using Gm = DeltaGeom<kD>;
  const long long rows = static_cast<long long>(a.B) * a.Hq * a.Lq;
  const long long rows_per_block = static_cast<long long>(Gm::THREADS / 32) * Gm::ROWS_PER_WARP * Gm::UNROLL;
  long long blocks = (rows + rows_per_block - 1) / rows_per_block;
  const long long cap = static_cast<long long>(a.num_sms > 0 ? a.num_sms : 152) * 8;
  if (blocks > cap) blocks = cap;
  // behind the forward: its CTAs take the SMs the forward's last CTAs free
  return launch_dependent(attn_delta_kernel<kD, BF16>, dim3(static_cast<unsigned>(blocks)), Gm::THREADS, 0, a.stream,
                          static_cast<const void*>(a.o), static_cast<const void*>(a.dO), a.delta_out, rows);
}

}  // namespace inst_d<D>

using namespace GBATTN_CAT(inst_d, GBATTN_HEAD_DIM);

int GBATTN_CAT(launch_fwd_d, GBATTN_HEAD_DIM)(const AttnArgs& a) {
  if (a.bf16) return a.causal ? fwd_impl<true, true>(a) : fwd_impl<true, false>(a);
  return a.causal ? fwd_impl<false, true>(a) : fwd_impl<false, false>(a);
}

int GBATTN_CAT(launch_bwd_d, GBATTN_HEAD_DIM)(const AttnArgs& a) {
  if (a.bf16) return a.causal ? bwd_impl<true, true>(a) : bwd_impl<true, false>(a);
  return a.causal ? bwd_impl<false, true>(a) : bwd_impl<false, false>(a);
}

int GBATTN_CAT(launch_bwd_dq_d, GBATTN_HEAD_DIM)(const AttnArgs& a) {
  if (a.bf16) return a.causal ? dq_impl<true, true>(a) : dq_impl<true, false>(a);
  return a.causal ? dq_impl<false, true>(a) : dq_impl<false, false>(a);
}

int GBATTN_CAT(launch_bwd_dkv_d, GBATTN_HEAD_DIM)(const AttnArgs& a) {
  if (a.bf16) return a.causal ? dkv_all<true, true>(a) : dkv_all<true, false>(a);
  return a.causal ? dkv_all<false, true>(a) : dkv_all<false, false>(a);
}

int GBATTN_CAT(launch_delta_d, GBATTN_HEAD_DIM)(const AttnArgs& a) {
  return a.bf16 ? delta_impl<true>(a) : delta_impl<false>(a);
}

int GBATTN_CAT(launch_fwd_decode_d, GBATTN_HEAD_DIM)(const AttnArgs& a) {
  if (a.bf16) return a.causal ? fwd_decode_impl<true, true>(a) : fwd_decode_impl<true, false>(a);
  return a.causal ? fwd_decode_impl<false, true>(a) : fwd_decode_impl<false, false>(a);
}

int GBATTN_CAT(launch_bwd_dkv_decode_d, GBATTN_HEAD_DIM)(const AttnArgs& a) {
  if (a.bf16) return a.causal ? dkv_decode_impl<true, true>(a) : dkv_decode_impl<true, false>(a);
  return a.causal ? dkv_decode_impl<false, true>(a) : dkv_decode_impl<false, false>(a);
}

int GBATTN_CAT(launch_bwd_dq_decode_d, GBATTN_HEAD_DIM)(const AttnArgs& a) {
  if (a.bf16) return a.causal ? dq_decode_impl<true, true>(a) : dq_decode_impl<true, false>(a);
  return a.causal ? dq_decode_impl<false, true>(a) : dq_decode_impl<false, false>(a);
}

}  // namespace gbattn
