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
// Decode layout (tcgen05 operand B for M <= kDecodeMaxM tokens).  K is padded
// with zeros to Kp = a multiple of 512; tokens are padded to Mt = M rounded up
// to 8.  The MMA's n dimension holds both planes of every token: row j < Mt is
// plane 0 of token j, row Mt + j plane 1 of token j.  Per k block of 128 inputs
// one contiguous block of 2 Mt rows x 128 bytes (256 Mt bytes), blocks in k
// order, so the operands of any run of k blocks are one contiguous range; inside
// a block the 16-byte chunk c of row r sits at chunk position c ^ (r % 8) (the
// 128-byte swizzle of the tensor core's shared-memory operands), and inside every
// group of 16 inputs the byte at position p holds input 16 g + pi(p), pi as in
// the prefill layout below.  Rows of tokens M..Mt-1 are never written and never
// reach a stored output.  Size: 2 * Mt * Kp bytes.
//
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

#include <stdint.h>

namespace bitlinear {

constexpr int kOpsBlockK = 512;
constexpr int64_t kDecodeMaxM = 32;      // more tokens: prefill layout and kernel

__host__ __device__ __forceinline__ bool act_ops_prefill(int64_t M) { return M > kDecodeMaxM; }

__host__ __device__ __forceinline__ int64_t act_ops_kpad(int64_t K) {
  return (K + kOpsBlockK - 1) / kOpsBlockK * kOpsBlockK;
}

__host__ __device__ __forceinline__ int64_t act_ops_mt(int64_t M) { return (M + 7) / 8 * 8; }

// Two small integers exact in e4m3 as two bytes, `lo` in the low byte (the PTX
// cvt to e4m3x2 puts its first source operand in the upper byte).  The ints
// become floats by the 1.5 * 2^23 offset (two full-rate operations) rather than
// a conversion instruction.
__device__ __forceinline__ uint32_t e4m3x2_exact(int lo, int hi) {
  const float fl = __fsub_rn(__int_as_float(lo + 0x4B400000), 12582912.0f);
  const float fh = __fsub_rn(__int_as_float(hi + 0x4B400000), 12582912.0f);
  unsigned short r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(fh), "f"(fl));
  return (uint32_t)r;
}

// Four words of e4m3 bytes of 16 consecutive codes in the pi order, for each
// plane; the codes come as int8 bytes, code j in byte j % 4 of q[j / 4].
__device__ __forceinline__ void act_ops_words(const uint32_t (&q)[4], uint32_t (&H)[4], uint32_t (&L)[4]) {
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    int hh[4], ll[4];
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const int pos = 4 * w + b;
      const int j = pos < 8 ? 2 * pos : 2 * (pos - 8) + 1;
      const int x = (int)(int8_t)(q[j >> 2] >> (8 * (j & 3)));
      const int h = (x + 8) >> 4;                 // arithmetic shift: floor
      hh[b] = 16 * h;
      ll[b] = x - 16 * h;
    }
    H[w] = e4m3x2_exact(hh[0], hh[1]) | (e4m3x2_exact(hh[2], hh[3]) << 16);
    L[w] = e4m3x2_exact(ll[0], ll[1]) | (e4m3x2_exact(ll[2], ll[3]) << 16);
  }
}

// Writes the operand bytes of 16 consecutive codes x_q[m][k..k+15], packed as
// int8 bytes in q (k a multiple of 16; zero codes for the padding beyond K), in
// the decode layout: two 16-byte stores, one per plane.
__device__ __forceinline__ void write_act_ops16(uint8_t* __restrict__ ops, int64_t M, int64_t m,
                                                int64_t k, int64_t Kp, const uint32_t (&q)[4]) {
  uint32_t H[4], L[4];
  act_ops_words(q, H, L);
  const int64_t Mt = act_ops_mt(M);
  const int64_t block = (k >> 7) * (256 * Mt);
  const int64_t c = (k >> 4) & 7, rh = m, rl = Mt + m;
  *reinterpret_cast<uint4*>(ops + block + rh * 128 + ((c ^ (rh & 7)) << 4)) = make_uint4(H[0], H[1], H[2], H[3]);
  *reinterpret_cast<uint4*>(ops + block + rl * 128 + ((c ^ (rl & 7)) << 4)) = make_uint4(L[0], L[1], L[2], L[3]);
  (void)Kp;
}

__host__ __device__ __forceinline__ int64_t act_ops_mpad(int64_t M) { return (M + 255) / 256 * 256; }

// Byte offset of the 16-byte chunk holding inputs [k, k + 16) of token m, plane 0.
__device__ __forceinline__ int64_t prefill_ops_offset(int64_t m, int64_t k, int64_t Kp) {
  const int64_t tt = m >> 8, r = m & 255, kb = k >> 7, c = (k >> 4) & 7;
  return ((tt * (Kp >> 7) + kb) << 15) + (r << 7) + ((c ^ (r & 7)) << 4);
}

// Prefill-layout counterpart of write_act_ops16.
__device__ __forceinline__ void write_act_ops16_prefill(uint8_t* __restrict__ ops, int64_t M, int64_t m,
                                                        int64_t k, int64_t Kp, const uint32_t (&q)[4]) {
  uint32_t H[4], L[4];
  act_ops_words(q, H, L);
  const int64_t off = prefill_ops_offset(m, k, Kp);
  *reinterpret_cast<uint4*>(ops + off) = make_uint4(H[0], H[1], H[2], H[3]);
  *reinterpret_cast<uint4*>(ops + act_ops_mpad(M) * Kp + off) = make_uint4(L[0], L[1], L[2], L[3]);
}

// Writes 16 codes in the layout that bitlinear_forward uses for M tokens.
__device__ __forceinline__ void write_act_ops16_any(uint8_t* __restrict__ ops, int64_t M, int64_t m,
                                                    int64_t k, int64_t Kp, const uint32_t (&q)[4]) {
  if (act_ops_prefill(M)) write_act_ops16_prefill(ops, M, m, k, Kp, q);
  else write_act_ops16(ops, M, m, k, Kp, q);
}

}  // namespace bitlinear
