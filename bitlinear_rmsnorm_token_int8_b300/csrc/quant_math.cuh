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

// element e (0..7, a compile-time index after unrolling) of eight packed bf16
__device__ __forceinline__ float bf16_at(const uint4& v, int e) {
  const uint32_t w = e < 2 ? v.x : e < 4 ? v.y : e < 6 ? v.z : v.w;
  return (e & 1) ? bf16_hi(w) : bf16_lo(w);
}

__device__ __forceinline__ void unpack8(const uint4& v, float (&f)[8]) {
  f[0] = bf16_lo(v.x); f[1] = bf16_hi(v.x);
  f[2] = bf16_lo(v.y); f[3] = bf16_hi(v.y);
  f[4] = bf16_lo(v.z); f[5] = bf16_hi(v.z);
  f[6] = bf16_lo(v.w); f[7] = bf16_hi(v.w);
}

// Rounding to an integer without the conversion pipe (which issues at a
// quarter of the FP32 rate): for |v| < 2^22, v + 1.5 * 2^23 lies where the fp32
// spacing is 1, so the round-to-nearest-even addition rounds v to an integer
// (ties to even), and that integer n sits in the low bits of the sum's encoding.
constexpr float kRoundMagic = 12582912.0f;   // 1.5 * 2^23, encoded 0x4B400000
__device__ __forceinline__ float rint_small(float v) { return __fsub_rn(__fadd_rn(v, kRoundMagic), kRoundMagic); }
// n as an int, for an integer-valued float |n| < 2^22
__device__ __forceinline__ int int_of_small(float n) { return __float_as_int(__fadd_rn(n, kRoundMagic)) - 0x4B400000; }

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
  float s;       // fl(127 / m) (small rows use fl(127 / c))
  float r;       // RMSNorm factor (used by small rows' codes)
  float sigma;   // dequantization factor of the row
  bool small;    // max|n| < 1e-8: the clamp applies
};

// Branch-free, so that the compiler can overlap this chain of IEEE operations
// with the codes of a regular row, which need only m and s.
__device__ __forceinline__ RowQuant row_quant(float m, float sum, int K, float rms_eps) {
  RowQuant q;
  const float rn = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(sum, (float)K), rms_eps)));
  q.r = rms_eps >= 0.0f ? rn : 1.0f;
  const float nmax = __fmul_rn(m, q.r);
  q.small = !(nmax >= kActClamp);
  q.m = m;
  q.s = __fdiv_rn(127.0f, m);
  q.sigma = q.small ? __fdiv_rn(kActClamp, 127.0f) : __fdiv_rn(nmax, 127.0f);
  return q;
}

// Codes of N inputs p(j) = x g of one row (N a multiple of 4; p: a callable,
// evaluated again for the rare inputs of the second pass instead of keeping N
// values live), packed as int8 bytes: code j is byte j % 4 of w[j / 4].  Each is
// the exactly rounded (ties to even) 127 p / m of a regular row (see the file
// comment), or the clamp's code of a small row.  t = p s (s = fl(127/m)) is
// within 2^-23 relative of 127 p / m and |t| < 127.5, so rint(t) is the code
// unless t lies within 2^-15 of a half-integer, i.e. |t - rint(t)| >= 1/2 - 2^-15
// (t - rint(t) is exact).  For those (about one input in 2^14) the sign of
// 127 p - (floor(t) + 1/2) m decides, formed by one fused multiply-add from the
// exact 127 p; an exact zero is a tie and goes to the even code.  The common
// path is a few full-rate operations per input and no branch, so a thread's
// inputs are independent chains; the low byte of rint(t) + 1.5 * 2^23's
// encoding is the code's two's-complement byte.
template <int N, typename P>
__device__ __forceinline__ void row_codes(P p, const RowQuant& rq, uint32_t (&w)[N / 4]) {
  float far = 0.0f;                          // largest |t - rint(t)|
#pragma unroll
  for (int g = 0; g < N / 4; ++g) {
    uint32_t b[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float t = __fmul_rn(p(4 * g + k), rq.s);
      const float mt = __fadd_rn(t, kRoundMagic);
      far = fmaxf(far, fabsf(__fsub_rn(t, __fsub_rn(mt, kRoundMagic))));
      b[k] = __float_as_uint(mt);
    }
    w[g] = __byte_perm(__byte_perm(b[0], b[1], 0x0040), __byte_perm(b[2], b[3], 0x0040), 0x5410);
  }
  if (rq.small) {
    // |p r| <= max|n| < 1e-8, so |t| < 127 and the clamp never acts
    const float sc = __fdiv_rn(127.0f, kActClamp);
#pragma unroll
    for (int g = 0; g < N / 4; ++g) {
      uint32_t b[4];
#pragma unroll
      for (int k = 0; k < 4; ++k)
        b[k] = (uint32_t)int_of_small(
            fminf(fmaxf(rint_small(__fmul_rn(__fmul_rn(p(4 * g + k), rq.r), sc)), -128.0f), 127.0f));
      w[g] = __byte_perm(__byte_perm(b[0], b[1], 0x0040), __byte_perm(b[2], b[3], 0x0040), 0x5410);
    }
  } else if (far >= 0.499969482421875f) {    // 1/2 - 2^-15: some input is near a half-integer
#pragma unroll
    for (int j = 0; j < N; ++j) {
      const float pj = p(j);
      const float t = __fmul_rn(pj, rq.s);
      const float rt = rint_small(t);
      if (fabsf(__fsub_rn(t, rt)) >= 0.499969482421875f) {
        const float f = rt > t ? __fsub_rn(rt, 1.0f) : rt;      // floor(t)
        const float h = __fadd_rn(f, 0.5f);                    // exact: |f| <= 127
        const float d = __fmaf_rn(-h, rq.m, __fmul_rn(127.0f, pj));
        const float up = __fadd_rn(f, 1.0f);
        const int c = int_of_small(d > 0.0f ? up : (d < 0.0f ? f : ((int_of_small(f) & 1) == 0 ? f : up)));
        const int sh = 8 * (j & 3);
        w[j >> 2] = (w[j >> 2] & ~(0xffu << sh)) | ((uint32_t)(c & 0xff) << sh);
      }
    }
  }
}

}  // namespace bitlinear
