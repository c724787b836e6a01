// Activation operands of the tensor-core contraction ("x_ops").
//
// An int8 code x in [-127, 127] is not exact in e4m3 (3 mantissa bits), but
// it splits exactly into two values that are:
//   h' = floor((x + 8) / 16) in [-8, 8],  l' = x - 16 h' in [-8, 7],
//   x = 16 h' + l',  and 16 h' and l' are both exact e4m3 numbers.
// A ternary weight is exact in e4m3 too, so W . x = W . (16 h) + W . l is two
// e4m3 tensor-core products into one fp32 accumulator, exact while the partial
// sums stay below 2^24 (|acc| <= 127 K).
//
// Decode layout (mma.sync m16n8k32 fragments, tokens in the n dimension).
// K is padded with zeros to Kp = a multiple of 512; tokens come in tiles of
// 16 (z = m / 16, mm = m % 16, Mz = min(16, M - 16 z) tokens in tile z).  The
// decode kernel reads the weights of a 512-wide k segment as one 128-byte
// swizzled row chunk, thread t of a quad taking k in [128 t, 128 t + 128) as
// two halves h of 64 k, four 16-k words j each.  For token m and index k:
//   seg = k / 512, t = (k % 512) / 128, h = (k % 128) / 64, j = (k % 64) / 16,
//   q = k % 16, u = 2 seg + h, i = 2 j + (q % 2), r = q / 8, pos = (q % 8) / 2,
//   byte = 32 Kp z + (((u * 8 + i) * Mz + mm) * 4 + t) * 16 + plane * 8 + r * 4 + pos,
// plane 0 = e4m3(16 h'), plane 1 = e4m3(l').  Thread t then loads the 16 bytes
// {H.b0, H.b1, L.b0, L.b1} of one k32 slab with one 16-byte load; the even/odd
// order inside each 4-byte register matches how the decode kernel unpacks the
// 2-bit weight codes (see decode_mma.cu).  The operands of one unit u of one
// token tile are contiguous (512 Mz bytes), so one bulk copy stages a run of
// units.  Size: 2 * M * Kp bytes.
// Prefill layout (tcgen05 operand B, tokens in the n dimension), used when
// M > kDecodeMaxM.  Tokens in tiles of 256 (Mp = M rounded up to 256), inputs
// in blocks of 128 (Kp as above).  Per (plane, token tile, k block) one
// contiguous 32 KB block of 256 rows x 128 bytes, blocks ordered plane-major,
// then token tile, then k block; inside a block the 16-byte chunk c of row r
// sits at chunk position c ^ (r % 8) (the 128-byte swizzle of the tensor core's
// shared-memory operands, so one bulk copy stages a block as the MMA reads it),
// and inside every group of 16 inputs the byte at position p holds input
// 16 g + pi(p), pi = (0, 2, 4, 6, 8, 10, 12, 14, 1, 3, 5, 7, 9, 11, 13, 15): the
// even inputs, then the odd ones, the order in which the prefill kernel writes
// decoded weights into tensor memory.  Plane 0 = 16 h', plane 1 = l'.  Rows of
// the last tile past M are never read into a stored output and are left as
// they are.  Size: 2 * Mp * Kp bytes.
#pragma once

#include <cuda_fp8.h>
#include <stdint.h>

namespace bitlinear {

constexpr int kOpsBlockK = 512;
constexpr int64_t kDecodeMaxM = 32;      // more tokens: prefill layout and kernel

__host__ __device__ __forceinline__ bool act_ops_prefill(int64_t M) { return M > kDecodeMaxM; }

__host__ __device__ __forceinline__ int64_t act_ops_kpad(int64_t K) {
  return (K + kOpsBlockK - 1) / kOpsBlockK * kOpsBlockK;
}

__device__ __forceinline__ uint32_t e4m3_exact(int v) {
  return (uint32_t)__nv_cvt_float_to_fp8((float)v, __NV_SATFINITE, __NV_E4M3);
}

// Writes the operand bytes of 16 consecutive codes q[0..15] = x_q[m][k..k+15]
// (k a multiple of 16; zero codes for the padding beyond K): two 16-byte stores.
__device__ __forceinline__ void write_act_ops16(uint8_t* __restrict__ ops, int64_t M, int64_t m,
                                                int64_t k, int64_t Kp, const int (&q)[16]) {
  const int64_t z = m >> 4, mm = m & 15;
  const int64_t Mz = (M - 16 * z) < 16 ? (M - 16 * z) : 16;
  const int64_t u = 2 * (k >> 9) + ((k >> 6) & 1);
  const int t = (int)(k >> 7) & 3, j = (int)(k >> 4) & 3;
#pragma unroll
  for (int p = 0; p < 2; ++p) {
    uint32_t H0 = 0, H1 = 0, L0 = 0, L1 = 0;
#pragma unroll
    for (int pos = 0; pos < 4; ++pos) {
      const int x0 = q[2 * pos + p], x1 = q[8 + 2 * pos + p];
      const int h0 = (x0 + 8) >> 4, h1 = (x1 + 8) >> 4;     // arithmetic shift: floor
      H0 |= e4m3_exact(16 * h0) << (8 * pos);
      L0 |= e4m3_exact(x0 - 16 * h0) << (8 * pos);
      H1 |= e4m3_exact(16 * h1) << (8 * pos);
      L1 |= e4m3_exact(x1 - 16 * h1) << (8 * pos);
    }
    const int64_t off = 32 * Kp * z + (((u * 8 + 2 * j + p) * Mz + mm) * 4 + t) * 16;
    *reinterpret_cast<uint4*>(ops + off) = make_uint4(H0, H1, L0, L1);
  }
}

__host__ __device__ __forceinline__ int64_t act_ops_mpad(int64_t M) { return (M + 255) / 256 * 256; }

// Byte offset of the 16-byte chunk holding inputs [k, k + 16) of token m, plane 0.
__device__ __forceinline__ int64_t prefill_ops_offset(int64_t m, int64_t k, int64_t Kp) {
  const int64_t tt = m >> 8, r = m & 255, kb = k >> 7, c = (k >> 4) & 7;
  return ((tt * (Kp >> 7) + kb) << 15) + (r << 7) + ((c ^ (r & 7)) << 4);
}

// Prefill-layout counterpart of write_act_ops16.
__device__ __forceinline__ void write_act_ops16_prefill(uint8_t* __restrict__ ops, int64_t M, int64_t m,
                                                        int64_t k, int64_t Kp, const int (&q)[16]) {
  uint32_t H[4], L[4];
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    H[w] = 0u;
    L[w] = 0u;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const int pos = 4 * w + b;
      const int x = q[pos < 8 ? 2 * pos : 2 * (pos - 8) + 1];
      const int h = (x + 8) >> 4;
      H[w] |= e4m3_exact(16 * h) << (8 * b);
      L[w] |= e4m3_exact(x - 16 * h) << (8 * b);
    }
  }
  const int64_t off = prefill_ops_offset(m, k, Kp);
  *reinterpret_cast<uint4*>(ops + off) = make_uint4(H[0], H[1], H[2], H[3]);
  *reinterpret_cast<uint4*>(ops + act_ops_mpad(M) * Kp + off) = make_uint4(L[0], L[1], L[2], L[3]);
}

// Writes 16 codes in the layout that bitlinear_forward uses for M tokens.
__device__ __forceinline__ void write_act_ops16_any(uint8_t* __restrict__ ops, int64_t M, int64_t m,
                                                    int64_t k, int64_t Kp, const int (&q)[16]) {
  if (act_ops_prefill(M)) write_act_ops16_prefill(ops, M, m, k, Kp, q);
  else write_act_ops16(ops, M, m, k, Kp, q);
}

}  // namespace bitlinear
