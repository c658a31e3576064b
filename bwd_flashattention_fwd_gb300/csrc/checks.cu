// libgbattn_checks.so: device-side checks of the attention kernels' own
// helpers, for the tests.  Not part of the attention interface.
//
//   gbattn_check_ex2_poly2(x, y, n, stream): y[i] = ex2_poly2(x[i]) for n
//   floats in device memory, evaluated with the same inline code the dQ and
//   dK/dV kernels use (ptx.cuh), so a test can hold it to its stated error
//   bound.  Returns 0 on launch, else the CUDA error code.
//   gbattn_check_index(status, first, count, extent, site, stream): one thread
//   runs the debug build's index check (kernel_common.cuh, compiled here with
//   the checks on) on [first, first + count) against [0, extent); a failed
//   check records its code in the int at `status` (device memory).  The check
//   only decides: no memory at those indices is touched.
#include <cuda_runtime.h>

#define GBATTN_DEBUG_CHECKS 1
#include "kernel_common.cuh"

namespace gbattn {
namespace checks {

__global__ void ex2_poly2_kernel(const float* __restrict__ x, float* __restrict__ y, int n) {
  const int i = 2 * (blockIdx.x * blockDim.x + threadIdx.x);
  if (i >= n) return;
  const float x0 = x[i];
  const float x1 = i + 1 < n ? x[i + 1] : 0.f;
  float y0, y1;
  ex2_poly2(x0, x1, y0, y1);
  y[i] = y0;
  if (i + 1 < n) y[i + 1] = y1;
}

__global__ void index_kernel(int* status, unsigned long long first, unsigned long long count,
                             unsigned long long extent, int site) {
  dbg_in_range(first, count, extent, status, site);
}

}  // namespace checks
}  // namespace gbattn

extern "C" int gbattn_check_ex2_poly2(const float* x, float* y, int n, cudaStream_t stream) {
  if (n <= 0) return 0;
  const int pairs = (n + 1) / 2;
  gbattn::checks::ex2_poly2_kernel<<<(pairs + 255) / 256, 256, 0, stream>>>(x, y, n);
  return static_cast<int>(cudaPeekAtLastError());
}

extern "C" int gbattn_check_index(int* status, unsigned long long first, unsigned long long count,
                                  unsigned long long extent, int site, cudaStream_t stream) {
  gbattn::checks::index_kernel<<<1, 1, 0, stream>>>(status, first, count, extent, site);
  return static_cast<int>(cudaPeekAtLastError());
}
