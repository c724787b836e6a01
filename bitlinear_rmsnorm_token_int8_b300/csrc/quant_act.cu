// Fused RMSNorm + per-token absmax int8 activation quantization.
//
// Page "BitNet b1.58 in Production: 1-Bit LLMs and Energy Benchmarks":
//   section "The Mathematical Mechanism", item 2 (absmax, Q_b = 127, per token),
//   item 4 (the activation scale max|x|/Q_b enters the dequantization), and
//   bit_linear.py BitLinear.forward (nn.RMSNorm before activation_quant).
//
// One CTA per token row.  The row is read once from HBM with 16-byte loads and
// kept in registers; a block reduction gives max|x*g| (exact: max is order
// free) and sum x^2 (fp32 pairwise inside a thread, fp64 across threads).
//
// Codes.  r > 0 is one number per row, so Round(127 n/max|n|) with n = x*r*g
// equals Round(127 p/max|p|) with p = x*g, and p is exact in fp32 (two 8-bit
// significands).  The kernel forms t = p * fl(127/m) (relative error <= 2^-23,
// i.e. |t - 127p/m| < 1.6e-5) and takes rint(t) unless t lies within 2^-15 of
// a half-integer; there it decides exactly in fp64, where 127*p and
// (floor(t)+0.5)*m are both exact products, with ties going to the even code.
#include <cuda_runtime.h>
#include <stdint.h>

#include "internal.h"

namespace bitlinear {
namespace {

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ void unpack8(const uint4& v, float (&f)[8]) {
  f[0] = bf16_lo(v.x); f[1] = bf16_hi(v.x);
  f[2] = bf16_lo(v.y); f[3] = bf16_hi(v.y);
  f[4] = bf16_lo(v.z); f[5] = bf16_hi(v.z);
  f[6] = bf16_lo(v.w); f[7] = bf16_hi(v.w);
}

// Exactly rounded code of 127*p/m (ties to even), see the file comment.
__device__ __forceinline__ int quant_code(float p, float s, float m) {
  const float t = __fmul_rn(p, s);
  const float f = floorf(t);
  const float dist = fabsf(__fsub_rn(t, __fadd_rn(f, 0.5f)));
  float q;
  if (dist > 3.0517578125e-05f) {          // 2^-15
    q = rintf(t);
  } else {
    const double a = 127.0 * (double)p;     // exact
    const double h = ((double)f + 0.5) * (double)m;  // exact: 9-bit * 24-bit
    if (a > h) q = f + 1.0f;
    else if (a < h) q = f;
    else q = (fmodf(f, 2.0f) == 0.0f) ? f : f + 1.0f;
  }
  q = fminf(fmaxf(q, -128.0f), 127.0f);
  return (int)q;
}

// eight bf16 ones
__device__ __constant__ uint4 kOnes = {0x3f803f80u, 0x3f803f80u, 0x3f803f80u, 0x3f803f80u};

template <int VPT>
__global__ void __launch_bounds__(1024)
quant_act_kernel(const uint4* __restrict__ x, const uint4* __restrict__ gain, float rms_eps,
                 int K, int8_t* __restrict__ x_q, float* __restrict__ act_scale) {
  const int V = K >> 3;                      // 16-byte vectors per row
  const int row = blockIdx.x;
  const int tid = threadIdx.x;
  const int T = blockDim.x;
  const uint4* xr = x + (size_t)row * V;

  uint4 xv[VPT];
  float amax = 0.0f;
  float part[VPT];
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    const int v = tid + i * T;
    part[i] = 0.0f;
    if (v < V) {
      xv[i] = __ldg(xr + v);
      float xf[8], gf[8];
      unpack8(xv[i], xf);
      unpack8(gain ? __ldg(gain + v) : kOnes, gf);
      float sq[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        amax = fmaxf(amax, fabsf(__fmul_rn(xf[j], gf[j])));
        sq[j] = __fmul_rn(xf[j], xf[j]);
      }
      part[i] = __fadd_rn(__fadd_rn(__fadd_rn(sq[0], sq[1]), __fadd_rn(sq[2], sq[3])),
                          __fadd_rn(__fadd_rn(sq[4], sq[5]), __fadd_rn(sq[6], sq[7])));
    }
  }
  // pairwise sum of the thread's vectors
#pragma unroll
  for (int w = 1; w < VPT; w <<= 1)
#pragma unroll
    for (int i = 0; i + w < VPT; i += 2 * w) part[i] = __fadd_rn(part[i], part[i + w]);
  double ss = (double)part[0];

  // block reduction: max (exact) and sum of squares (fp64)
  __shared__ float s_max[32];
  __shared__ double s_ss[32];
  __shared__ float s_m;
  __shared__ double s_sum;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    ss += __shfl_xor_sync(0xffffffffu, ss, o);
  }
  const int lane = tid & 31, warp = tid >> 5, nwarps = T >> 5;
  if (lane == 0) { s_max[warp] = amax; s_ss[warp] = ss; }
  __syncthreads();
  if (warp == 0) {
    float a = lane < nwarps ? s_max[lane] : 0.0f;
    double s = lane < nwarps ? s_ss[lane] : 0.0;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
      s += __shfl_xor_sync(0xffffffffu, s, o);
    }
    if (lane == 0) { s_m = a; s_sum = s; }
  }
  __syncthreads();

  const float m = fmaxf(s_m, 1e-8f);
  const float s = __fdiv_rn(127.0f, m);
  if (tid == 0) {
    double sigma = (double)m / 127.0;
    if (rms_eps >= 0.0f) sigma = sigma / sqrt(s_sum / (double)K + (double)rms_eps);
    act_scale[row] = (float)sigma;
  }

  uint2* qr = reinterpret_cast<uint2*>(x_q + (size_t)row * K);
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    const int v = tid + i * T;
    if (v < V) {
      float xf[8], gf[8];
      unpack8(xv[i], xf);
      unpack8(gain ? __ldg(gain + v) : kOnes, gf);
      uint32_t lo = 0, hi = 0;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        lo |= (uint32_t)(quant_code(__fmul_rn(xf[j], gf[j]), s, m) & 0xff) << (8 * j);
        hi |= (uint32_t)(quant_code(__fmul_rn(xf[j + 4], gf[j + 4]), s, m) & 0xff) << (8 * j);
      }
      qr[v] = make_uint2(lo, hi);
    }
  }
}

}  // namespace

cudaError_t launch_quant_act(const uint16_t* x, const uint16_t* gain, float rms_eps, int64_t M,
                             int64_t K, int8_t* x_q, float* act_scale, cudaStream_t stream) {
  if (M == 0) return cudaSuccess;
  const int V = (int)(K / 8);
  int T, vpt;
  if (V <= 256) {
    T = ((V + 31) / 32) * 32;
    vpt = 1;
  } else if (V <= 2048) {
    T = 256;
    vpt = (V + 255) / 256;
  } else {
    T = 1024;
    vpt = (V + 1023) / 1024;
  }
  int tv = 1;
  while (tv < vpt) tv <<= 1;
  const dim3 grid((unsigned)M), block((unsigned)T);
  const uint4* xv = reinterpret_cast<const uint4*>(x);
  const uint4* gv = reinterpret_cast<const uint4*>(gain);
  switch (tv) {
    case 1: quant_act_kernel<1><<<grid, block, 0, stream>>>(xv, gv, rms_eps, (int)K, x_q, act_scale); break;
    case 2: quant_act_kernel<2><<<grid, block, 0, stream>>>(xv, gv, rms_eps, (int)K, x_q, act_scale); break;
    case 4: quant_act_kernel<4><<<grid, block, 0, stream>>>(xv, gv, rms_eps, (int)K, x_q, act_scale); break;
    default: quant_act_kernel<8><<<grid, block, 0, stream>>>(xv, gv, rms_eps, (int)K, x_q, act_scale); break;
  }
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace bitlinear
