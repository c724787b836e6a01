// Per-tensor absmax int8 quantization with Q_b = 128, the scale-granularity
// variant of page "BitNet 1-bit LLM Inference Framework", BitLinear.
// activation_quantize: one scale for the whole tensor,
//   gamma = max_{t,k} |x|,  x_q = Round(Clip(x * 128 / (gamma + 1e-8), -128, 127)),
// the clip before the rounding as the page's code does (codes in [-128, 127]),
// and the dequant factor gamma / 2^7 for every token.  No RMSNorm: that page's
// BitLinear quantizes its input directly.
//
// Two kernels: row_absmax_kernel writes max|x| of every row to scratch;
// per_tensor_codes_kernel (a programmatic dependent of the first) reduces those
// maxima to gamma in every CTA (max is order free, so all CTAs agree) and codes
// the rows.  Each code is decided on the binary32 quotient fl(fl(x * 128) / d),
// d = fl(gamma + 1e-8): x * 128 is exact and __fdiv_rn rounds once, as the
// page's binary32 tensors do.
#include <cuda_runtime.h>
#include <stdint.h>

#include "act_ops.cuh"
#include "device_util.cuh"
#include "internal.h"
#include "quant_math.cuh"

namespace bitlinear {
namespace {

constexpr int kPtThreads = 256;

// Block-wide max of non-negative values; every thread gets the result.
__device__ __forceinline__ float block_max(float a, float* s_red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
  if ((threadIdx.x & 31) == 0) s_red[threadIdx.x >> 5] = a;
  __syncthreads();
  a = 0.0f;
#pragma unroll
  for (int w = 0; w < kPtThreads / 32; ++w) a = fmaxf(a, s_red[w]);
  __syncthreads();                           // s_red may be reused
  return a;
}

__global__ void __launch_bounds__(kPtThreads)
row_absmax_kernel(const uint4* __restrict__ x, int64_t M, int V, float* __restrict__ row_max) {
  __shared__ float s_red[kPtThreads / 32];
  pdl_launch_dependents();                   // the codes kernel waits for this one to complete
  pdl_wait();                                // x may be the previous kernel's output
  for (int64_t row = blockIdx.x; row < M; row += gridDim.x) {
    float a = 0.0f;
    for (int v = threadIdx.x; v < V; v += kPtThreads) {
      float xf[8];
      unpack8(__ldcg(x + row * V + v), xf);
#pragma unroll
      for (int j = 0; j < 8; ++j) a = fmaxf(a, fabsf(xf[j]));
    }
    a = block_max(a, s_red);
    if (threadIdx.x == 0) row_max[row] = a;
  }
}

__global__ void __launch_bounds__(kPtThreads)
per_tensor_codes_kernel(const uint4* __restrict__ x, int64_t M, int K, const float* __restrict__ row_max,
                        int8_t* __restrict__ x_q, float* __restrict__ act_scale, uint8_t* __restrict__ x_ops) {
  __shared__ float s_red[kPtThreads / 32];
  pdl_launch_dependents();
  pdl_wait();                                // row_max is the previous kernel's output
  float g = 0.0f;
  for (int64_t i = threadIdx.x; i < M; i += kPtThreads) g = fmaxf(g, __ldcg(row_max + i));
  g = block_max(g, s_red);
  const float d = __fadd_rn(g, 1e-8f);
  const float sigma = __fmul_rn(g, 0.0078125f);  // gamma / 2^7, exact
  const int V = K >> 3;
  const int64_t Kp = act_ops_kpad(K);
  for (int64_t row = blockIdx.x; row < M; row += gridDim.x) {
    if (threadIdx.x == 0) act_scale[row] = sigma;
    uint2* qr = x_q ? reinterpret_cast<uint2*>(x_q + row * K) : nullptr;
    for (int u = threadIdx.x; u < (int)(Kp >> 4); u += kPtThreads) {
      uint32_t w[4];
#pragma unroll
      for (int hv = 0; hv < 2; ++hv) {
        const int v = 2 * u + hv;
        w[2 * hv] = w[2 * hv + 1] = 0u;              // padding up to Kp: zero operands
        if (v < V) {
          float xf[8];
          unpack8(__ldcg(x + row * V + v), xf);
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const float t = fminf(fmaxf(__fdiv_rn(__fmul_rn(xf[j], 128.0f), d), -128.0f), 127.0f);
            w[2 * hv + (j >> 2)] |= (uint32_t)((int)rintf(t) & 0xff) << (8 * (j & 3));
          }
          if (qr) qr[v] = make_uint2(w[2 * hv], w[2 * hv + 1]);
        }
      }
      if (x_ops) write_act_ops16_any(x_ops, M, row, (int64_t)u << 4, Kp, w);
    }
  }
}

}  // namespace

cudaError_t launch_quant_act_per_tensor(const uint16_t* x, int64_t M, int64_t K, int8_t* x_q, float* act_scale,
                                        uint8_t* x_ops, float* row_max, bool pdl, cudaStream_t stream) {
  if (M == 0) return cudaSuccess;
  const int64_t cap = (int64_t)num_sms() * 8;
  const unsigned grid = (unsigned)(M < cap ? M : cap);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(kPtThreads, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  const uint4* xv = reinterpret_cast<const uint4*>(x);
  cudaError_t e = cudaLaunchKernelEx(&cfg, row_absmax_kernel, xv, M, (int)(K / 8), row_max);
  if (e != cudaSuccess) return e;
  cfg.numAttrs = 1;                          // the second kernel follows ours: overlap is safe
  e = cudaLaunchKernelEx(&cfg, per_tensor_codes_kernel, xv, M, (int)K, (const float*)row_max, x_q, act_scale,
                         x_ops);
  count_launches(2);
  return e;
}

}  // namespace bitlinear
