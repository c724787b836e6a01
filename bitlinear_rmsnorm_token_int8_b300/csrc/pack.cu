// Absmean ternarization and 2-bit packing of latent weights.
//
// Page "BitNet b1.58 in Production: 1-Bit LLMs and Energy Benchmarks", section
// "The Mathematical Mechanism", item 1 (gamma = mean|W|, W_q = Clip(Round(W /
// (gamma + eps)), -1, 1)); page "BitNet 1-bit LLM Inference Framework", section
// "How the LUT Kernel Works" (code 00 = 0, 01 = +1, 10 = -1, four per byte).
//
// gamma is the exact mean of |W| rounded once to binary32, so it does not
// depend on how the sum is split across threads:
//   1. absmean_bins: every |w| = mant24 * 2^(e-150) (normal) or mant * 2^-149
//      (subnormal).  The kernel adds each mantissa into a 64-bit integer bin of
//      its exponent (shared-memory bins per CTA, then global atomics).  Integer
//      adds are associative, so the bins are exact and order free.
//   2. gamma_finalize (one thread): sums the bins into a base-2^32 multi-digit
//      integer (units of 2^-149), divides by N*K with a long division, and
//      rounds the quotient to binary32 (nearest, ties to even) from the
//      quotient bits, a round bit and a sticky bit.
//   3. ternarize_pack: W_q = sign(W) where 2|W| > d = fl32(gamma + eps), else 0,
//      written in the tile-major layout of the contraction kernels (internal.h).
//      This is exactly Round(W/d) clipped to [-1, 1]: |W/d| = 1/2 is a tie that
//      rounds to the even value 0, and every |W/d| > 1/2 rounds to a non-zero
//      integer that the clip maps to sign(W).  2|W| is exact in binary32.
#include <cuda_runtime.h>
#include <stdint.h>

#include "internal.h"

namespace bitlinear {
namespace {

constexpr int kBinsThreads = 256;

__global__ void __launch_bounds__(kBinsThreads)
absmean_bins_kernel(const float4* __restrict__ w4, int64_t n4, unsigned long long* __restrict__ bins,
                    int* __restrict__ dev_err) {
  __shared__ unsigned long long s_bins[256];
  for (int i = threadIdx.x; i < 256; i += blockDim.x) s_bins[i] = 0ull;
  __syncthreads();
  bool bad = false;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4;
       i += (int64_t)gridDim.x * blockDim.x) {
    const float4 v = __ldg(w4 + i);
    const float f[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t bits = __float_as_uint(f[j]) & 0x7fffffffu;
      const uint32_t e = bits >> 23;
      uint32_t mant = bits & 0x7fffffu;
      if (e == 255u) { bad = true; continue; }
      if (bits == 0u) continue;
      if (e != 0u) mant |= 0x800000u;
      atomicAdd(&s_bins[e], (unsigned long long)mant);
    }
  }
  if (bad) atomicCAS(dev_err, 0, kDevErrNonFinite);
  __syncthreads();
  for (int i = threadIdx.x; i < 256; i += blockDim.x)
    if (s_bins[i]) atomicAdd(&bins[i], s_bins[i]);
}

// The exact mean S / count rounded once to binary32 (nearest, ties to even), where
// S = sum_e bins[e] * 2^(max(e,1)-1) in units of 2^-149 (count < 2^32).  One thread.
__device__ float exact_mean_f32(const unsigned long long* bins, uint64_t count) {
  constexpr int L = 16;                      // 512 bits: S < 2^342, then shifted by 64
  uint32_t s[L];
#pragma unroll
  for (int i = 0; i < L; ++i) s[i] = 0u;
  for (int e = 0; e < 255; ++e) {
    const unsigned long long b = bins[e];     // < 2^56
    if (b == 0ull) continue;
    const int pos = (e > 0 ? e : 1) - 1 + 64; // +64: S * 2^64 so the quotient keeps fraction bits
    const int limb = pos >> 5, off = pos & 31;
    // b << off spans at most three base-2^32 digits
    const uint64_t sh = b << off;
    const uint64_t add[3] = {sh & 0xffffffffull, sh >> 32, off ? (b >> (64 - off)) : 0ull};
    uint64_t carry = 0;
    for (int j = 0; limb + j < L && (j < 3 || carry); ++j) {
      const uint64_t t = (uint64_t)s[limb + j] + (j < 3 ? add[j] : 0ull) + carry;
      s[limb + j] = (uint32_t)t;
      carry = t >> 32;
    }
  }
  // Q = floor(S * 2^64 / count), R = remainder (count < 2^32)
  uint32_t q[L];
  uint64_t rem = 0;
  for (int i = L - 1; i >= 0; --i) {
    const uint64_t cur = (rem << 32) | s[i];
    q[i] = (uint32_t)(cur / count);
    rem = cur % count;
  }
  int top = -1;
  for (int i = L - 1; i >= 0; --i)
    if (q[i]) { top = i; break; }
  float gamma;
  if (top < 0) {
    gamma = 0.0f;                             // S == 0 (S > 0 gives Q >= 2^32)
  } else {
    const int b = top * 32 + (32 - __clz(q[top]));   // bit length of Q
    // value = Q * 2^-213; keep bits down to 2^-149 (Q bit 64) for subnormals
    const int shift = (b - 24 > 64) ? (b - 24) : 64;
    auto bit = [&](int i) -> uint32_t { return (q[i >> 5] >> (i & 31)) & 1u; };
    uint32_t mant = 0;
    for (int i = b - 1; i >= shift; --i) mant = (mant << 1) | bit(i);
    const uint32_t rbit = bit(shift - 1);
    bool sticky = rem != 0;
    for (int i = 0; i < shift - 1 && !sticky; ++i) sticky = bit(i) != 0;
    if (rbit && (sticky || (mant & 1u))) ++mant;
    // mant in [2^23, 2^24] for normals (the 2^23 bit adds one to the exponent field)
    uint32_t bits = ((uint32_t)(shift - 64) << 23) + mant;
    if (bits >= 0x7f800000u) bits = 0x7f800000u;
    gamma = __uint_as_float(bits);
  }
  return gamma;
}

// One thread: gamma of the whole matrix and d = fl32(gamma + eps).
__global__ void gamma_finalize_kernel(const unsigned long long* __restrict__ bins, uint64_t count,
                                      float eps, float* __restrict__ gd, float* __restrict__ gamma_out) {
  if (threadIdx.x != 0 || blockIdx.x != 0) return;
  const float gamma = exact_mean_f32(bins, count);
  gd[0] = gamma;
  gd[1] = __fadd_rn(gamma, eps);
  if (gamma_out) *gamma_out = gamma;
}

// Per output channel: CTA n sums |W[n, :]| into exponent bins in shared memory
// (order free, as absmean_bins_kernel) and its thread 0 writes gamma_n, the exact
// row mean rounded once, to w_scale[n].  Rows n = blockIdx.x, blockIdx.x + gridDim.x, ...
__global__ void __launch_bounds__(kBinsThreads)
row_absmean_kernel(const float4* __restrict__ w4, int64_t N, int64_t K4, float* __restrict__ w_scale,
                   int* __restrict__ dev_err) {
  __shared__ unsigned long long s_bins[256];
  for (int64_t n = blockIdx.x; n < N; n += gridDim.x) {
    for (int i = threadIdx.x; i < 256; i += blockDim.x) s_bins[i] = 0ull;
    __syncthreads();
    bool bad = false;
    for (int64_t i = threadIdx.x; i < K4; i += blockDim.x) {
      const float4 v = __ldg(w4 + n * K4 + i);
      const float f[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t bits = __float_as_uint(f[j]) & 0x7fffffffu;
        const uint32_t e = bits >> 23;
        uint32_t mant = bits & 0x7fffffu;
        if (e == 255u) { bad = true; continue; }
        if (bits == 0u) continue;
        if (e != 0u) mant |= 0x800000u;
        atomicAdd(&s_bins[e], (unsigned long long)mant);
      }
    }
    if (bad) atomicCAS(dev_err, 0, kDevErrNonFinite);
    __syncthreads();
    if (threadIdx.x == 0) w_scale[n] = exact_mean_f32(s_bins, (uint64_t)(K4 * 4));
    __syncthreads();                          // thread 0 has read the bins before the next row clears them
  }
}

// One thread per 16-byte chunk of the tiled layout (64 weights of one row; see
// internal.h): codes of rows >= N or k >= K are 0.  One scale for the matrix (gd =
// gamma, fl32(gamma + eps); gamma is written to every w_scale[n]), or, with per_row,
// the row's own gamma_n read from w_scale[n] and d = fl32(gamma_n + eps).
__global__ void ternarize_pack_kernel(const float* __restrict__ W, int64_t N, int64_t K,
                                      int64_t nseg, int64_t chunks, int64_t Np, const float* __restrict__ gd,
                                      uint8_t* __restrict__ packed, float* __restrict__ w_scale, float eps,
                                      bool per_row) {
  const float gamma = per_row ? 0.0f : gd[0];
  float d = per_row ? 0.0f : gd[1];
  const int64_t full_tiles = Np / 128, tile_chunks = nseg * 128 * 8;   // chunks of a full tile
  for (int64_t ci = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; ci < chunks;
       ci += (int64_t)gridDim.x * blockDim.x) {
    int64_t t = ci / tile_chunks;
    if (t > full_tiles) t = full_tiles;                          // inside the last, partial tile
    const int64_t rows = (t < full_tiles) ? 128 : Np - 128 * full_tiles;
    const int64_t w = ci - t * tile_chunks;                      // chunk index within the tile
    const int64_t seg = w / (rows * 8);
    const int q = (int)(w - seg * rows * 8);
    const int r = q >> 3, c = (q & 7) ^ (r & 7);                 // row in the tile, logical chunk
    const int64_t n = t * 128 + r;
    const int64_t k0 = seg * 512 + c * 64;
    uint32_t out[4] = {0u, 0u, 0u, 0u};
    if (n < N) {
      if (per_row) d = __fadd_rn(w_scale[n], eps);
      const float* wr = W + n * K;
#pragma unroll 4
      for (int q = 0; q < 16; ++q) {             // 16 groups of four weights = 16 bytes
        const int64_t k = k0 + 4 * q;
        if (k < K) {
          const float4 v = __ldg(reinterpret_cast<const float4*>(wr + k));
          const float f[4] = {v.x, v.y, v.z, v.w};
          uint32_t byte = 0;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float a = __fmul_rn(2.0f, fabsf(f[j]));
            const uint32_t code = (a > d) ? (f[j] > 0.0f ? 1u : 2u) : 0u;
            byte |= code << (2 * j);
          }
          out[q >> 2] |= byte << (8 * (q & 3));
        }
      }
      if (seg == 0 && c == 0 && !per_row) w_scale[n] = gamma;
    }
    *reinterpret_cast<uint4*>(packed + (ci << 4)) = make_uint4(out[0], out[1], out[2], out[3]);
  }
}

}  // namespace

cudaError_t launch_pack_weights(const float* W, int64_t N, int64_t K, float eps, uint8_t* packed,
                                float* w_scale, float* gamma_out, void* workspace, int* dev_err,
                                cudaStream_t stream) {
  unsigned long long* bins = reinterpret_cast<unsigned long long*>(workspace);
  float* gd = reinterpret_cast<float*>(reinterpret_cast<char*>(workspace) + kPackBinsBytes);
  cudaError_t err = cudaMemsetAsync(workspace, 0, kPackWorkspaceBytes, stream);
  if (err != cudaSuccess) return err;
  const int64_t n4 = N * K / 4;
  const int sms = num_sms();
  int64_t blocks = (n4 + kBinsThreads - 1) / kBinsThreads;
  if (blocks > (int64_t)sms * 8) blocks = (int64_t)sms * 8;
  const float4* w4 = reinterpret_cast<const float4*>(W);
  absmean_bins_kernel<<<(unsigned)blocks, kBinsThreads, 0, stream>>>(w4, n4, bins, dev_err);
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  gamma_finalize_kernel<<<1, 32, 0, stream>>>(bins, (uint64_t)(N * K), eps, gd, gamma_out);
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  const int64_t nseg = packed_nseg(K);
  const int64_t chunks = packed_layout_bytes(N, K) / 16;
  int64_t pblocks = (chunks + 255) / 256;
  if (pblocks > (int64_t)sms * 16) pblocks = (int64_t)sms * 16;
  ternarize_pack_kernel<<<(unsigned)pblocks, 256, 0, stream>>>(W, N, K, nseg, chunks, packed_rows(N), gd, packed,
                                                               w_scale, eps, false);
  count_launches(3);
  return cudaGetLastError();
}

cudaError_t launch_pack_weights_per_channel(const float* W, int64_t N, int64_t K, float eps, uint8_t* packed,
                                            float* w_scale, int* dev_err, cudaStream_t stream) {
  const int sms = num_sms();
  const int64_t rblocks = N < (int64_t)sms * 8 ? N : (int64_t)sms * 8;
  row_absmean_kernel<<<(unsigned)rblocks, kBinsThreads, 0, stream>>>(reinterpret_cast<const float4*>(W), N, K / 4,
                                                                      w_scale, dev_err);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  const int64_t chunks = packed_layout_bytes(N, K) / 16;
  int64_t pblocks = (chunks + 255) / 256;
  if (pblocks > (int64_t)sms * 16) pblocks = (int64_t)sms * 16;
  ternarize_pack_kernel<<<(unsigned)pblocks, 256, 0, stream>>>(W, N, K, packed_nseg(K), chunks, packed_rows(N),
                                                               nullptr, packed, w_scale, eps, true);
  count_launches(2);
  return cudaGetLastError();
}

}  // namespace bitlinear
