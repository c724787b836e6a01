// Dispatch of bitlinear_forward to the contraction kernels.
#include <cuda_runtime.h>
#include <stdint.h>

#include "act_ops.cuh"
#include "internal.h"

namespace bitlinear {

// Scratch for converting x_q to the operand form; none when the codes kernel takes x_q.
size_t forward_workspace_bytes(int64_t M, int64_t N, int64_t K) {
  return codes_route(M, N, K) ? 0 : act_ops_bytes(M, K);
}

cudaError_t launch_forward(const int8_t* x_q, const float* act_scale, const uint8_t* x_ops,
                           const uint8_t* packed, const float* w_scale, int64_t M, int64_t N,
                           int64_t K, int out_dtype, void* y, int32_t* acc_debug, void* workspace,
                           int* dev_err, bool pdl, cudaStream_t stream, L2Prefetch pf) {
  // a few tokens with their int8 codes at hand: the CUDA-core kernel, which needs no
  // operand form
  if (x_q && codes_route(M, N, K))
    return launch_codes_cc(x_q, act_scale, packed, w_scale, M, N, K, out_dtype, y, acc_debug, pdl, stream, pf);
  if (!x_ops) {
    uint8_t* ops = static_cast<uint8_t*>(workspace);
    cudaError_t e = launch_act_ops_from_codes(x_q, M, K, ops, pdl, stream);
    if (e != cudaSuccess) return e;
    x_ops = ops;
    pdl = true;   // the operand kernel just enqueued is ours: overlap with it is safe
  }
  // the prefill contraction is bound by its tensor cores, not by its weight stream:
  // it takes no prefetch
  if (act_ops_prefill(M))
    return launch_prefill_tc(x_ops, act_scale, packed, w_scale, M, N, K, out_dtype, y, acc_debug,
                             dev_err, pdl, stream);
  return launch_decode_tc(x_ops, act_scale, packed, w_scale, M, N, K, out_dtype, y, acc_debug,
                          dev_err, pdl, stream, pf);
}

}  // namespace bitlinear
