// Scalar steps of the RMSNorm + absmax int8 quantization shared by the
// quantization kernels and the fused one-token layer kernel, so that both
// compute the same codes and scale bit for bit (see quant_act.cu for the
// arithmetic and its error bounds).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace bitlinear {

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
    const float a = __fmul_rn(127.0f, p);                       // exact
    const float d = __fmaf_rn(-__fadd_rn(f, 0.5f), m, a);       // sign of 127p - (f+1/2)m
    if (d > 0.0f) q = f + 1.0f;
    else if (d < 0.0f) q = f;
    else q = (fmodf(f, 2.0f) == 0.0f) ? f : f + 1.0f;
  }
  q = fminf(fmaxf(q, -128.0f), 127.0f);
  return (int)q;
}

// Error-free sum of two fp32 numbers: s + e == a + b exactly (Knuth).
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
  s = __fadd_rn(a, b);
  const float bb = __fsub_rn(s, a);
  e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}

// (h1 + l1) + (h2 + l2) as a renormalised pair.
__device__ __forceinline__ void pair_add(float& h1, float& l1, float h2, float l2) {
  float s, e;
  two_sum(h1, h2, s, e);
  e = __fadd_rn(e, __fadd_rn(l1, l2));
  h1 = __fadd_rn(s, e);
  l1 = __fsub_rn(e, __fsub_rn(h1, s));
}

// eight bf16 ones
static __device__ __constant__ uint4 kOnes = {0x3f803f80u, 0x3f803f80u, 0x3f803f80u, 0x3f803f80u};


// Block-wide max and pair sum of the per-thread (amax, hi + lo), in a fixed order:
// an xor tree within each warp, then warp 0 over the warps' partials (zero for
// warps past nwarps), the same tree again.  s_max / s_ss: 32 entries each.
__device__ __forceinline__ void block_stats(float amax, float hi, float lo, int tid, int nwarps, float* s_max,
                                            float2* s_ss, float* s_m, float* s_sum) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float h2 = __shfl_xor_sync(0xffffffffu, hi, o), l2 = __shfl_xor_sync(0xffffffffu, lo, o);
    pair_add(hi, lo, h2, l2);
  }
  const int lane = tid & 31, warp = tid >> 5;
  if (lane == 0) { s_max[warp] = amax; s_ss[warp] = make_float2(hi, lo); }
  __syncthreads();
  if (warp == 0) {
    float a = lane < nwarps ? s_max[lane] : 0.0f;
    float2 p2 = lane < nwarps ? s_ss[lane] : make_float2(0.0f, 0.0f);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
      const float h2 = __shfl_xor_sync(0xffffffffu, p2.x, o), l2 = __shfl_xor_sync(0xffffffffu, p2.y, o);
      pair_add(p2.x, p2.y, h2, l2);
    }
    if (lane == 0) { *s_m = a; *s_sum = __fadd_rn(p2.x, p2.y); }
  }
  __syncthreads();
}

// activation_quant's clamp of the normalized row's max|n|, n = x r g
constexpr float kActClamp = 1e-8f;

// The per-row constants of the quantization, formed identically by every
// thread from the row's max|x g| (m, exact) and fl32 sum of x^2.
//   r     = fl(1 / fl(sqrt(fl(fl(sum / K) + eps))))   (1 without RMSNorm)
//   max|n| = fl(m r); a row with max|n| >= 1e-8 quantizes on p = x g with
//   s = fl(127 / m) (r cancels from n / max|n|) and sigma = fl(max|n| / 127);
//   a row below the clamp ("small") has c = 1e-8: codes rint(fl(fl(p r) fl(127 / c)))
//   and sigma = fl(c / 127).
struct RowQuant {
  float m;       // max|p| (regular rows)
  float s;       // fl(127 / m), or fl(127 / c) for small rows
  float r;       // RMSNorm factor (used by small rows' codes)
  float sigma;   // dequantization factor of the row
  bool small;    // max|n| < 1e-8: the clamp applies
};

__device__ __forceinline__ RowQuant row_quant(float m, float sum, int K, float rms_eps) {
  RowQuant q;
  q.r = 1.0f;
  if (rms_eps >= 0.0f) q.r = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(sum, (float)K), rms_eps)));
  const float nmax = __fmul_rn(m, q.r);
  q.small = !(nmax >= kActClamp);
  q.m = m;
  if (!q.small) {
    q.s = __fdiv_rn(127.0f, m);
    q.sigma = __fdiv_rn(nmax, 127.0f);
  } else {
    q.s = __fdiv_rn(127.0f, kActClamp);
    q.sigma = __fdiv_rn(kActClamp, 127.0f);
  }
  return q;
}

// Code of input p = x g of a row with constants q.
__device__ __forceinline__ int row_code(float p, const RowQuant& q) {
  if (!q.small) return quant_code(p, q.s, q.m);
  const float t = __fmul_rn(__fmul_rn(p, q.r), q.s);
  return (int)fminf(fmaxf(rintf(t), -128.0f), 127.0f);
}

}  // namespace bitlinear
