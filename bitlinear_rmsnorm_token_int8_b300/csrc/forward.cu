// Dispatch of bitlinear_forward to the contraction kernels.
#include <cuda_runtime.h>
#include <stdint.h>

#include "internal.h"

namespace bitlinear {

cudaError_t launch_gemv_dp4a(const int8_t* x_q, const float* act_scale, const uint8_t* packed,
                             const float* w_scale, int64_t M, int64_t N, int64_t K, int out_dtype,
                             void* y, int32_t* acc_debug, cudaStream_t stream);

size_t forward_workspace_bytes(int64_t, int64_t, int64_t) { return 0; }

cudaError_t launch_forward(const int8_t* x_q, const float* act_scale, const uint8_t* packed,
                           const float* w_scale, int64_t M, int64_t N, int64_t K, int out_dtype,
                           void* y, int32_t* acc_debug, void*, int*, cudaStream_t stream) {
  // token tiles of at most 65535 * 8 rows per launch (grid.y limit)
  const int64_t max_tokens = 65535LL * 8;
  for (int64_t t0 = 0; t0 < M; t0 += max_tokens) {
    const int64_t m = (M - t0 < max_tokens) ? (M - t0) : max_tokens;
    const size_t esz = out_dtype == 0 ? 4 : 2;
    cudaError_t e = launch_gemv_dp4a(x_q + t0 * K, act_scale + t0, packed, w_scale, m, N, K, out_dtype,
                                     static_cast<char*>(y) + (size_t)t0 * N * esz,
                                     acc_debug ? acc_debug + t0 * N : nullptr, stream);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace bitlinear
