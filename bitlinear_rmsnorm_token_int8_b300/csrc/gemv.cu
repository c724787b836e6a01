// Ternary contraction on the CUDA cores: int8 tokens x 2-bit packed weights,
// exact int32 accumulation with dp4a, fused dequantization.
//
// Page "BitNet b1.58 in Production: 1-Bit LLMs and Energy Benchmarks", section
// "The Mathematical Mechanism", items 3-4; page "BitNet 1-bit LLM Inference
// Framework", section "How the LUT Kernel Works" (2-bit code, int32 accumulate).
//
// A weight of +1, 0 or -1 times an int8 activation is an add, a skip or a
// subtract; dp4a does four of them at once on int8 lanes holding the decoded
// weights (0x01, 0x00, 0xFF), so acc is exact (|acc| <= 127 K < 2^31).
//
// Layout of the work: a warp owns 8 weight rows; lane = 4*r + c reads 16-byte
// chunk c, c+4, c+8, ... of row r (64 weights per chunk, coalesced 64-byte runs
// per row) and accumulates up to 8 tokens; the 4 lanes of a row are reduced
// with shuffles.  blockIdx.y walks tiles of 8 tokens.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "internal.h"

namespace bitlinear {
namespace {

constexpr int kTileTokens = 8;
constexpr int kWarps = 4;
constexpr int kRowsPerWarp = 8;

// 2-bit codes of one byte-pair spread to one code per nibble.
__device__ __forceinline__ uint32_t spread_codes(uint32_t h16) {
  uint32_t t = h16 & 0xffffu;
  t = (t | (t << 8)) & 0x00ff00ffu;
  t = (t | (t << 4)) & 0x0f0f0f0fu;
  t = (t | (t << 2)) & 0x33333333u;
  return t;
}

// byte table for __byte_perm: code 0 -> 0x00, 1 -> 0x01 (+1), 2 -> 0xFF (-1)
constexpr uint32_t kCodeToInt8 = 0x00ff0100u;

__device__ __forceinline__ void decode16(uint32_t w, int (&o)[4]) {
  const uint32_t lo = spread_codes(w), hi = spread_codes(w >> 16);
  o[0] = (int)__byte_perm(kCodeToInt8, 0u, lo);
  o[1] = (int)__byte_perm(kCodeToInt8, 0u, lo >> 16);
  o[2] = (int)__byte_perm(kCodeToInt8, 0u, hi);
  o[3] = (int)__byte_perm(kCodeToInt8, 0u, hi >> 16);
}

__global__ void __launch_bounds__(kWarps * 32)
gemv_dp4a_kernel(const int8_t* __restrict__ x_q, const float* __restrict__ act_scale,
                 const uint8_t* __restrict__ packed, const float* __restrict__ w_scale, int M, int N,
                 int K, int out_dtype, void* __restrict__ y, int32_t* __restrict__ acc_debug) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int r = lane >> 2, c = lane & 3;
  const int row = (blockIdx.x * kWarps + warp) * kRowsPerWarp + r;
  const int t0 = blockIdx.y * kTileTokens;
  const int nt = min(kTileTokens, M - t0);
  const int chunks = K >> 6;
  int acc[kTileTokens];
#pragma unroll
  for (int t = 0; t < kTileTokens; ++t) acc[t] = 0;
  if (row < N) {
    const uint4* wrow = reinterpret_cast<const uint4*>(packed + (size_t)row * (K >> 2));
    for (int kc = c; kc < chunks; kc += 4) {
      const uint4 wv = __ldg(wrow + kc);
      int wd[16];
      {
        int o[4];
        decode16(wv.x, o); wd[0] = o[0]; wd[1] = o[1]; wd[2] = o[2]; wd[3] = o[3];
        decode16(wv.y, o); wd[4] = o[0]; wd[5] = o[1]; wd[6] = o[2]; wd[7] = o[3];
        decode16(wv.z, o); wd[8] = o[0]; wd[9] = o[1]; wd[10] = o[2]; wd[11] = o[3];
        decode16(wv.w, o); wd[12] = o[0]; wd[13] = o[1]; wd[14] = o[2]; wd[15] = o[3];
      }
#pragma unroll
      for (int t = 0; t < kTileTokens; ++t) {
        if (t < nt) {
          const int4* xr = reinterpret_cast<const int4*>(x_q + (size_t)(t0 + t) * K + ((size_t)kc << 6));
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int4 xv = __ldg(xr + j);
            acc[t] = __dp4a(wd[4 * j + 0], xv.x, acc[t]);
            acc[t] = __dp4a(wd[4 * j + 1], xv.y, acc[t]);
            acc[t] = __dp4a(wd[4 * j + 2], xv.z, acc[t]);
            acc[t] = __dp4a(wd[4 * j + 3], xv.w, acc[t]);
          }
        }
      }
    }
  }
#pragma unroll
  for (int t = 0; t < kTileTokens; ++t) {
    acc[t] += __shfl_xor_sync(0xffffffffu, acc[t], 1);
    acc[t] += __shfl_xor_sync(0xffffffffu, acc[t], 2);
  }
  if (row < N && c == 0) {
    const float ws = w_scale[row];
#pragma unroll
    for (int t = 0; t < kTileTokens; ++t) {
      if (t < nt) {
        const size_t o = (size_t)(t0 + t) * N + row;
        const float v = __fmul_rn(__fmul_rn((float)acc[t], act_scale[t0 + t]), ws);
        if (out_dtype == 0) reinterpret_cast<float*>(y)[o] = v;
        else reinterpret_cast<__nv_bfloat16*>(y)[o] = __float2bfloat16_rn(v);
        if (acc_debug) acc_debug[o] = acc[t];
      }
    }
  }
}

}  // namespace

cudaError_t launch_gemv_dp4a(const int8_t* x_q, const float* act_scale, const uint8_t* packed,
                             const float* w_scale, int64_t M, int64_t N, int64_t K, int out_dtype,
                             void* y, int32_t* acc_debug, cudaStream_t stream) {
  const int rows_per_cta = kWarps * kRowsPerWarp;
  const dim3 grid((unsigned)((N + rows_per_cta - 1) / rows_per_cta),
                  (unsigned)((M + kTileTokens - 1) / kTileTokens));
  gemv_dp4a_kernel<<<grid, kWarps * 32, 0, stream>>>(x_q, act_scale, packed, w_scale, (int)M, (int)N,
                                                      (int)K, out_dtype, y, acc_debug);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace bitlinear
