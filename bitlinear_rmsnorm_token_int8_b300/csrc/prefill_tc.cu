// Prefill contraction (many tokens) on the 5th-generation tensor cores:
// y = dequant(x_q . W_q^T) with tcgen05.mma kind::f8f6f4, accumulators in
// tensor memory (TMEM).
//
// Page "BitNet b1.58 in Production: 1-Bit LLMs and Energy Benchmarks", section
// "The Mathematical Mechanism", items 3-4; page "BitNet 1-bit LLM Inference
// Framework", section "How the LUT Kernel Works" (2-bit code, int32 sums).
// The method's integer contraction is a dense matmul once M is large, so it is
// run as one: this GPU has no int8 tcgen05 MMA, so each int8 code enters as two
// exact e4m3 values (16 h' + l', act_ops.cuh) against e4m3 weights of -1/0/+1,
// two MMAs per k step into one fp32 accumulator, exact while every partial sum
// stays below 2^24 in magnitude (at most 128 K + 8 K <= 2^23 + 2^19 for codes
// in [-128, 127] and K <= 65536).
//
// Tile: 128 weight rows (MMA M, operand A) x TT = 256 or 128 tokens (MMA N,
// operand B), persistent clusters of CL = 1 or 2 CTAs over tiles (TMA multicast
// of the activation planes within a cluster, see prefill_tc_kernel).
// 128-token tiles double the number of tiles where 256-token ones would leave
// many SMs idle (a few hundred tokens, or a last wave at most half full); the
// operand layout is the same (a 128-token tile reads half of a 256-token block).
// Roles (512 threads, warpgroup-aligned so that setmaxnreg can move registers
// from the producer and decoder warpgroups to the epilogue ones):
//   warp 0      weight producer: per 512-k segment, one bulk copy of the tile's
//               packed weights (up to 16 KB, the tile-major layout).
//   warp 2      operand producer: per 128-k step, one bulk copy per operand plane
//               of the token tile's block (or half), already in the swizzled
//               layout the MMA reads (act_ops.cuh).  Two threads, so that neither
//               ring waits for the other's slots (one thread serving both held
//               the operand copies behind the weight ring: 8B down 148 -> 143 us
//               with two).  Copies are few and large because the copy engine's
//               cost is per request, and per 128-byte row for tensor-map boxes.
//   warp 1      allocates TMEM (512 columns: D = TT, A = 2 x 128 at 256) and
//               issues the MMAs, per 128-k step 4 k32 steps x 2 planes: the whole
//               warp runs the loop and one elected lane issues.
//   warp 3      idle (the rest of the first warpgroup).
//   warps 4-7   decoders: thread = weight row; 2-bit codes -> e4m3 bytes by
//               byte permutes, written to TMEM as the A operand (tcgen05.st),
//               128 columns per segment, double buffered.
//   warps 8-15  epilogue: two warps per TMEM lane quarter (warpgroups 2 and 3),
//               each taking half of the tile's tokens.  A warp loads all its
//               accumulators (tcgen05.ld, up to 4 x 32 columns) into registers
//               and releases them at once, so that the MMAs of the next tile run
//               while it forms y = fl(fl(acc * act_scale[m]) * w_scale[n]) and
//               stores (measured: the MMA warp had stalled about 6 us per tile
//               for an epilogue that held the accumulators through its stores).
// Weights reach the tensor core through TMEM rather than shared memory: the
// decode expands 2 bits to 8, and TMEM takes those writes without costing
// shared-memory bandwidth.
//
// A row's codes are decoded word by word (16 codes): the four TMEM columns of a
// word hold the weights of inputs (0,2,4,6), (8..14 even), (1,3,5,7), (9..15
// odd); the prefill operand layout stores the activations in that order.
//
// Every mbarrier wait is bounded: on expiry the kernel records
// BITLINEAR_ERR_TIMEOUT, all roles stop, MMAs and copies in flight are waited
// for (bounded), and TMEM is freed before the CTA exits.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "act_ops.cuh"
#include "device_util.cuh"
#include "internal.h"

namespace bitlinear {
namespace {

constexpr int kTileW = 128;                 // weight rows per tile (MMA M)
constexpr int kBlockT = 256;                // tokens per block of the operand layout
constexpr int kThreads = 512;               // four warpgroups (see the roles above)
// Registers per thread of each warpgroup after setmaxnreg: the launch gives every
// thread 128 (the kernel is compiled to exactly that, checked before launch), and
// the split must not exceed that total (128 x (56 + 104) + 256 x 176 = 512 x 128).
constexpr uint32_t kRegsCtl = 56, kRegsDec = 104, kRegsEpi = 176;
static_assert(128 * (kRegsCtl + kRegsDec) + 256 * kRegsEpi == kThreads * 128, "register split");
constexpr int kNSXMax = 6;                  // operand stages (128 k each): 3 x 64 KB or 6 x 32 KB
constexpr int kNSW = 2;                     // weight stages (512 k each)
constexpr int kXBytes = 3 * 2 * kBlockT * 128;  // 192 KB of operand stages for either tile
constexpr int kWStageBytes = 128 * 128;     // one segment: 128 rows x 128 bytes of packed codes
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColA = 256;             // A buffers at columns 256 and 384
constexpr uint32_t kSpin = 1u << 24;
constexpr uint32_t kCodeToE4M3 = 0x00B83800u;  // bytes 0x00 (code 0), 0x38 (+1), 0xB8 (-1)

// shared memory (after 1024-byte alignment)
constexpr int kOffX = 0;
constexpr int kOffW = kOffX + kXBytes;
constexpr int kOffBar = kOffW + kNSW * kWStageBytes;
constexpr int kNumBars = 2 * kNSXMax + 2 * kNSW + 2 * 2 + 2 + 1;
constexpr int kSmemBytes = 1024 + kOffBar + kNumBars * 8 + 16;

struct PrefillParams {
  const uint8_t* packed;
  const uint8_t* x_ops;
  int64_t plane_bytes;            // Mp * Kp
  const float* act_scale;
  const float* w_scale;
  void* y;
  int32_t* acc_debug;
  int* dev_err;
  int M, N, K, out_dtype;
  int nseg, ntiles_n16, nwb, ntok, tiles;
};

struct Bars {
  uint32_t full_x, empty_x, full_w, empty_w, a_full, a_empty, d_full, d_empty, fin;
};

template <int NSX>
__device__ __forceinline__ Bars bars_at(uint32_t base) {
  Bars b;
  b.full_x = base;
  b.empty_x = b.full_x + 8 * NSX;
  b.full_w = b.empty_x + 8 * NSX;
  b.empty_w = b.full_w + 8 * kNSW;
  b.a_full = b.empty_w + 8 * kNSW;
  b.a_empty = b.a_full + 16;
  b.d_full = b.a_empty + 16;
  b.d_empty = b.d_full + 8;
  b.fin = b.d_empty + 8;
  return b;
}

// Bounded wait; on expiry records the error and raises the CTA's abort flag.
__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                              int* dev_err) {
  if (mbar_wait_bounded(bar, parity, kSpin)) return true;
  atomicCAS(dev_err, 0, kDevErrTimeout);
  *abort_flag = 1;
  return false;
}

// Warp-collective form for the warps whose next step is a tcgen05 load or
// store (.sync.aligned): every lane takes the same branch.
__device__ __forceinline__ bool warp_wait_or_abort(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                                   int* dev_err) {
  const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(bar, parity, kSpin));
  if (!ok && (threadIdx.x & 31) == 0) {
    atomicCAS(dev_err, 0, kDevErrTimeout);
    *abort_flag = 1;
  }
  __syncwarp();
  return ok;
}

__device__ __forceinline__ bool warp_aborted(volatile int* abort_flag) {
  return __any_sync(0xffffffffu, *abort_flag != 0);
}

// CL CTAs of a cluster work on CL neighbouring weight blocks of the same token
// tile: each copies 256 / CL token rows of every operand stage and multicasts
// them to all CL, and each one's MMA completion releases the stage in all CL,
// so the cluster reads the activations from L2 once instead of CL times.
template <int CL, int TT>
__global__ void __launch_bounds__(kThreads, 1) prefill_tc_kernel(const PrefillParams p) {
  constexpr int kNSX = 3 * kBlockT / TT;        // operand stages
  constexpr int kXPlaneBytes = TT * 128;        // one plane of a stage: TT token rows x 128 k
  constexpr int kXStageBytes = 2 * kXPlaneBytes;
  constexpr int kTilesPerBlock = kBlockT / TT;  // token tiles per block of the operand layout
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  __shared__ uint32_t s_tmem;
  __shared__ volatile int s_abort;
  const uint32_t sbase = smem_u32(smem);
  const Bars B = bars_at<kNSX>(sbase + kOffBar);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kNSX; ++s) {
      mbar_init(B.full_x + 8 * s, 1);
      mbar_init(B.empty_x + 8 * s, CL);            // one MMA commit from each CTA of the cluster
    }
    for (int s = 0; s < kNSW; ++s) {
      mbar_init(B.full_w + 8 * s, 1);
      mbar_init(B.empty_w + 8 * s, 4);            // the four decoder warps
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(B.a_full + 8 * s, 4);
      mbar_init(B.a_empty + 8 * s, 1);
    }
    mbar_init(B.d_full, 1);
    mbar_init(B.d_empty, 8);                      // the eight epilogue warps
    mbar_init(B.fin, 1);
    s_abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(smem_u32(&s_tmem), kTmemCols);
  tc_fence_before();
  __syncthreads();
  if (CL > 1) cluster_sync();                      // peers' barriers exist before any multicast
  tc_fence_after();
  pdl_launch_dependents();
  const uint32_t tmem = s_tmem;
  const int nseg = p.nseg;
  const int rank = CL > 1 ? (int)cluster_ctarank() : 0;
  const int cid = blockIdx.x / CL, ncl = gridDim.x / CL;
  const int nwbg = (p.nwb + CL - 1) / CL;          // weight-block groups
  const int ctiles = nwbg * p.ntok;
  constexpr uint16_t kMask = (uint16_t)((1u << CL) - 1);

  // Each warpgroup's branch starts with its register count: fewer for the
  // producer/MMA and decoder warpgroups, more for the epilogue's.
  if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsCtl));
    if (warp == 0) {
      // ------------------------------------------------------------ weight producer
      // The packed weights are not written by earlier kernels: no dependency wait.
      if (lane == 0) {
        int ws = 0;
        for (int ct = cid; ct < ctiles && !s_abort; ct += ncl) {
          const int wb = (ct % nwbg) * CL + rank;
          for (int sg = 0; sg < nseg && !s_abort; ++sg) {
            const int wslot = ws % kNSW, wround = ws / kNSW;
            if (wround >= 1 && !wait_or_abort(B.empty_w + 8 * wslot, (wround - 1) & 1, &s_abort, p.dev_err))
              break;
            // the tile's rows of this segment: one contiguous block of the packed layout
            const int rows = max(0, min(128, 16 * p.ntiles_n16 - wb * 128));
            mbar_arrive_expect_tx(B.full_w + 8 * wslot, (uint32_t)(rows * 128));
            if (rows > 0)
              bulk_g2s(sbase + kOffW + wslot * kWStageBytes,
                       p.packed + (int64_t)wb * nseg * 16384 + (int64_t)sg * rows * 128, (uint32_t)(rows * 128),
                       B.full_w + 8 * wslot);
            ++ws;
          }
        }
        // nothing may still be landing in shared memory when the CTA exits
        for (int s = 0; s < kNSW && s < ws; ++s) {
          const int last = ws - 1 - ((ws - 1 - s) % kNSW);
          if (!mbar_wait_bounded(B.full_w + 8 * s, (last / kNSW) & 1, kSpin)) atomicCAS(p.dev_err, 0, kDevErrTimeout);
        }
      }
    } else if (warp == 2) {
      // ------------------------------------------------------------ operand producer
      // Its own thread, so that the operand ring runs ahead of the weight ring.
      if (lane == 0) {
        pdl_wait();                                  // operands come from the previous kernel
        int xs = 0;
        for (int ct = cid; ct < ctiles && !s_abort; ct += ncl) {
          const int tt = ct / nwbg;
          const int blk = tt / kTilesPerBlock, sub = tt % kTilesPerBlock;
          for (int sg = 0; sg < nseg && !s_abort; ++sg) {
            for (int kk = 0; kk < 4; ++kk) {
              const int xslot = xs % kNSX, xround = xs / kNSX;
              if (xround >= 1 && !wait_or_abort(B.empty_x + 8 * xslot, (xround - 1) & 1, &s_abort, p.dev_err))
                break;
              mbar_arrive_expect_tx(B.full_x + 8 * xslot, (uint32_t)kXStageBytes);
              const uint32_t part = kXPlaneBytes / CL;            // this CTA's rows of the block
              const uint32_t dst = sbase + kOffX + xslot * kXStageBytes + rank * part;
              const uint8_t* src = p.x_ops + (((int64_t)blk * (nseg * 4) + sg * 4 + kk) << 15) +
                                   sub * kXPlaneBytes + rank * part;
              if (CL > 1) {
                bulk_g2s_mc(dst, src, part, B.full_x + 8 * xslot, kMask);
                bulk_g2s_mc(dst + kXPlaneBytes, src + p.plane_bytes, part, B.full_x + 8 * xslot, kMask);
              } else {
                bulk_g2s(dst, src, part, B.full_x + 8 * xslot);
                bulk_g2s(dst + kXPlaneBytes, src + p.plane_bytes, part, B.full_x + 8 * xslot);
              }
              ++xs;
            }
          }
        }
        for (int s = 0; s < kNSX && s < xs; ++s) {
          const int last = xs - 1 - ((xs - 1 - s) % kNSX);
          if (!mbar_wait_bounded(B.full_x + 8 * s, (last / kNSX) & 1, kSpin)) atomicCAS(p.dev_err, 0, kDevErrTimeout);
        }
      }
    } else if (warp == 1) {
      // ------------------------------------------------------------ MMA issue
      // The whole warp runs the loop (warp-uniform waits and descriptors); one
      // elected lane, the same throughout, issues every MMA and commit.
      const uint32_t idesc = idesc_e4m3_f32(kTileW, TT);
      int xs = 0, as = 0, tcount = 0;
      auto aborted = [&]() { return __any_sync(0xffffffffu, s_abort != 0); };
      for (int ct = cid; ct < ctiles && !aborted(); ct += ncl, ++tcount) {
        if (tcount >= 1 && !warp_wait_or_abort(B.d_empty, (tcount - 1) & 1, &s_abort, p.dev_err)) break;
        tc_fence_after();
        bool first = true;
        for (int sg = 0; sg < nseg && !aborted(); ++sg) {
          const int ab = as & 1;
          if (!warp_wait_or_abort(B.a_full + 8 * ab, (as >> 1) & 1, &s_abort, p.dev_err)) break;
          tc_fence_after();
          for (int kk = 0; kk < 4; ++kk) {
            const int xslot = xs % kNSX;
            if (!warp_wait_or_abort(B.full_x + 8 * xslot, (xs / kNSX) & 1, &s_abort, p.dev_err)) break;
            tc_fence_after();
            const uint32_t xh = sbase + kOffX + xslot * kXStageBytes, xl = xh + kXPlaneBytes;
#pragma unroll
            for (int s = 0; s < 4; ++s) {
              const uint32_t a = tmem + kColA + ab * 128 + kk * 32 + s * 8;
              if (elect_one()) {
                mma_f8f6f4_ts(tmem, a, smem_desc_sw128(xh + 32 * s), idesc, first ? 0u : 1u);
                mma_f8f6f4_ts(tmem, a, smem_desc_sw128(xl + 32 * s), idesc, 1u);
              }
              __syncwarp();
              first = false;
            }
            if (elect_one()) {
              if (CL > 1) mma_commit_mc(B.empty_x + 8 * xslot, kMask);   // frees the stage in every CTA
              else mma_commit(B.empty_x + 8 * xslot);
            }
            __syncwarp();
            ++xs;
          }
          if (elect_one()) mma_commit(B.a_empty + 8 * ab);           // frees the A buffer
          __syncwarp();
          ++as;
        }
        if (elect_one()) mma_commit(B.d_full);                       // accumulators complete
        __syncwarp();
      }
      // before TMEM is freed every MMA issued here must be finished
      if (elect_one()) mma_commit(B.fin);
      __syncwarp();
      if (lane == 0 && !mbar_wait_bounded(B.fin, 0, kSpin)) atomicCAS(p.dev_err, 0, kDevErrTimeout);
      __syncwarp();
    }
  } else if (warp < 8) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsDec));
    // ------------------------------------------------------------ decoders
    const int q4 = warp & 3;                   // TMEM lane quarter of this warp
    const int r = 32 * q4 + lane;              // weight row within the block
    const uint32_t lane_addr = (uint32_t)(32 * q4) << 16;
    int ws = 0, as = 0;
    for (int ct = cid; ct < ctiles && !warp_aborted(&s_abort); ct += ncl) {
      const int wb = (ct % nwbg) * CL + rank;
      const bool valid = wb * kTileW + r < p.N;
      for (int sg = 0; sg < nseg; ++sg) {
        const int wslot = ws % kNSW, ab = as & 1;
        if (!warp_wait_or_abort(B.full_w + 8 * wslot, (ws / kNSW) & 1, &s_abort, p.dev_err)) break;
        if (as >= 2 && !warp_wait_or_abort(B.a_empty + 8 * ab, ((as >> 1) - 1) & 1, &s_abort, p.dev_err)) break;
        tc_fence_after();
        // row r of the stage: line r; chunk c stored at c ^ (r % 8)
        const uint32_t row = sbase + kOffW + wslot * kWStageBytes + r * 128;
#pragma unroll
        for (int cp = 0; cp < 4; ++cp) {        // chunk pairs: 32 TMEM columns each
          uint32_t cols[32];
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) {
            const int c = 2 * cp + cc;
            const uint4 v = valid ? lds128(row + (uint32_t)((c ^ (r & 7)) << 4)) : make_uint4(0u, 0u, 0u, 0u);
            const uint32_t wd[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const uint32_t lo = wd[j] & 0x33333333u, hi = (wd[j] >> 2) & 0x33333333u;
              uint32_t* o = cols + 16 * cc + 4 * j;
              o[0] = __byte_perm(kCodeToE4M3, 0u, lo);          // inputs 0, 2, 4, 6
              o[1] = __byte_perm(kCodeToE4M3, 0u, lo >> 16);    // 8, 10, 12, 14
              o[2] = __byte_perm(kCodeToE4M3, 0u, hi);          // 1, 3, 5, 7
              o[3] = __byte_perm(kCodeToE4M3, 0u, hi >> 16);    // 9, 11, 13, 15
            }
          }
          tmem_st32(tmem + lane_addr + kColA + ab * 128 + cp * 32, cols);
        }
        tmem_wait_st();
        __syncwarp();
        if (lane == 0) mbar_arrive(B.empty_w + 8 * wslot);   // weight stage read
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(B.a_full + 8 * ab);       // A buffer written
        ++ws;
        ++as;
      }
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsEpi));
    // ------------------------------------------------------------ epilogue
    pdl_wait();                                // act_scale and y follow the stream order
    const int q4 = warp & 3;
    const int half = (warp - 8) >> 2;          // tokens [TT/2 half, TT/2 (half + 1)) of the tile
    const uint32_t lane_addr = (uint32_t)(32 * q4) << 16;
    constexpr int kChunks = TT / 2 / 32;       // chunks of 32 tokens per warp
    const int out_mode = p.out_dtype;
    int tcount = 0;
    for (int ct = cid; ct < ctiles && !warp_aborted(&s_abort); ct += ncl, ++tcount) {
      const int wb = (ct % nwbg) * CL + rank, tt = ct / nwbg;
      const int n = wb * kTileW + 32 * q4 + lane;
      const bool nv = n < p.N;
      const float wsn = nv ? __ldg(p.w_scale + n) : 0.0f;
      const int m0 = tt * TT + half * (TT / 2);
      float as_lane[kChunks];
#pragma unroll
      for (int c = 0; c < kChunks; ++c) {
        const int m = m0 + 32 * c + lane;
        as_lane[c] = m < p.M ? __ldcg(p.act_scale + m) : 0.0f;
      }
      if (!warp_wait_or_abort(B.d_full, tcount & 1, &s_abort, p.dev_err)) break;
      tc_fence_after();
      uint32_t rv[kChunks][32];
#pragma unroll
      for (int c = 0; c < kChunks; ++c) tmem_ld32(tmem + lane_addr + half * (TT / 2) + 32 * c, rv[c]);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(B.d_empty);   // accumulators may be overwritten
#pragma unroll
      for (int c = 0; c < kChunks; ++c) {
        const int mbase = m0 + 32 * c;
        const int jmax = nv ? min(32, p.M - mbase) : 0;       // tokens of this chunk that exist
        const size_t o0 = (size_t)mbase * p.N + n;
        if (out_mode == 1) {                                 // bf16
          __nv_bfloat16* yb = reinterpret_cast<__nv_bfloat16*>(p.y) + o0;
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const float as = __shfl_sync(0xffffffffu, as_lane[c], j);
            if (j < jmax) yb[(size_t)j * p.N] = __float2bfloat16_rn(__fmul_rn(__fmul_rn(__uint_as_float(rv[c][j]), as), wsn));
          }
        } else if (out_mode == 0) {                          // fp32
          float* yf = reinterpret_cast<float*>(p.y) + o0;
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const float as = __shfl_sync(0xffffffffu, as_lane[c], j);
            if (j < jmax) yf[(size_t)j * p.N] = __fmul_rn(__fmul_rn(__uint_as_float(rv[c][j]), as), wsn);
          }
        } else {                                             // bf16 residual add
          __nv_bfloat16* yb = reinterpret_cast<__nv_bfloat16*>(p.y) + o0;
          // residuals 16 at a time, loaded before the stores: a load after a store to y
          // could not be moved ahead of it
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            float res[16];
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) {
              const int j = 16 * hh + jj;
              res[jj] = j < jmax ? __uint_as_float((uint32_t)__ldcg(reinterpret_cast<const unsigned short*>(yb) +
                                                                     (size_t)j * p.N) << 16)
                                 : 0.0f;
            }
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) {
              const int j = 16 * hh + jj;
              const float as = __shfl_sync(0xffffffffu, as_lane[c], j);
              if (j < jmax) {
                const float yv = __fmul_rn(__fmul_rn(__uint_as_float(rv[c][j]), as), wsn);
                yb[(size_t)j * p.N] = __float2bfloat16_rn(__fadd_rn(res[jj], yv));
              }
            }
          }
        }
        if (p.acc_debug) {
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (j < jmax) p.acc_debug[o0 + (size_t)j * p.N] = (int32_t)__uint_as_float(rv[c][j]);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (CL > 1) cluster_sync();                      // no peer still sends data or arrivals here
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

// True when p points into device memory of the calling thread's current device.
// Anything else (host memory, managed memory, a peer GPU's memory reached through
// unified addressing, or a pointer the runtime does not know) is not.
bool local_device_memory(const void* p) {
  int dev = -1;
  cudaPointerAttributes a = {};
  if (cudaGetDevice(&dev) != cudaSuccess || cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return a.type == cudaMemoryTypeDevice && a.device == dev;
}

// CTAs per cluster of the prefill contraction: 2 (the activation blocks multicast
// to both CTAs of a cluster; measured: 2 beats 1 and 4) when there are at least two
// weight blocks and the operands lie in the current device's own memory, so that a
// multicast copy only ever reads this GPU's memory; 1 otherwise.
int prefill_cluster(const void* x_ops, int64_t N) {
  const int64_t nwb = (N + kTileW - 1) / kTileW;
  return nwb >= 2 && local_device_memory(x_ops) ? 2 : 1;
}

// Tokens per tile: 128 when that takes less time in tile-rounds of the persistent
// grid, a 128-token tile costing 0.74 of a 256-token one (measured on B300 over
// 2B and 8B shapes at 256-2048 tokens: half the MMAs and operand bytes, but the
// same weight decode and a fixed cost per tile).
int prefill_tile_tokens(int64_t M, int64_t N, int CL, int sms) {
  const int64_t nwb = (N + kTileW - 1) / kTileW;
  const int64_t ncl = sms / CL > 0 ? sms / CL : 1;
  const int64_t g = (nwb + CL - 1) / CL;
  const int64_t r256 = (g * ((M + 255) / 256) + ncl - 1) / ncl;
  const int64_t r128 = (g * ((M + 127) / 128) + ncl - 1) / ncl;
  return 74 * r128 < 100 * r256 ? 128 : 256;
}

cudaError_t launch_prefill_tc(const uint8_t* x_ops, const float* act_scale, const uint8_t* packed,
                              const float* w_scale, int64_t M, int64_t N, int64_t K, int out_dtype,
                              void* y, int32_t* acc_debug, int* dev_err, bool pdl,
                              cudaStream_t stream) {
  const int64_t Kp = act_ops_kpad(K);
  const int64_t nwb = (N + kTileW - 1) / kTileW;
  const int CL = prefill_cluster(x_ops, N);
  const int sms = num_sms();
  const int TT = prefill_tile_tokens(M, N, CL, sms);
  PrefillParams p = {};
  p.packed = packed;
  p.x_ops = x_ops;
  p.plane_bytes = act_ops_mpad(M) * Kp;
  p.act_scale = act_scale;
  p.w_scale = w_scale;
  p.y = y;
  p.acc_debug = acc_debug;
  p.dev_err = dev_err;
  p.M = (int)M;
  p.N = (int)N;
  p.K = (int)K;
  p.out_dtype = out_dtype;
  p.nseg = (int)(Kp / 512);
  p.ntiles_n16 = (int)(N / 16);
  p.nwb = (int)((N + kTileW - 1) / kTileW);
  p.ntok = (int)((M + TT - 1) / TT);
  const int64_t tiles = (int64_t)p.nwb * p.ntok;
  if (tiles > (1LL << 30)) return cudaErrorInvalidValue;
  p.tiles = (int)tiles;
  static bool attr_set = false;
  if (!attr_set) {
    for (void* f : {(void*)prefill_tc_kernel<1, 256>, (void*)prefill_tc_kernel<2, 256>,
                    (void*)prefill_tc_kernel<1, 128>, (void*)prefill_tc_kernel<2, 128>}) {
      cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
      if (e != cudaSuccess) return e;
      // setmaxnreg moves registers within what the launch gave: 128 per thread
      cudaFuncAttributes fa;
      e = cudaFuncGetAttributes(&fa, f);
      if (e != cudaSuccess) return e;
      if (fa.numRegs != 128) return cudaErrorInvalidConfiguration;
    }
    attr_set = true;
  }
  const int64_t ctiles = ((nwb + CL - 1) / CL) * p.ntok;
  int64_t clusters = sms / CL;
  if (clusters > ctiles) clusters = ctiles;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(clusters * CL), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  int na = 0;
  attr[na].id = cudaLaunchAttributeClusterDimension;
  attr[na].val.clusterDim.x = (unsigned)CL;
  attr[na].val.clusterDim.y = 1;
  attr[na].val.clusterDim.z = 1;
  ++na;
  if (pdl) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  cudaError_t e;
  if (TT == 128) {
    if (CL == 2) e = cudaLaunchKernelEx(&cfg, prefill_tc_kernel<2, 128>, p);
    else e = cudaLaunchKernelEx(&cfg, prefill_tc_kernel<1, 128>, p);
  } else {
    if (CL == 2) e = cudaLaunchKernelEx(&cfg, prefill_tc_kernel<2, 256>, p);
    else e = cudaLaunchKernelEx(&cfg, prefill_tc_kernel<1, 256>, p);
  }
  count_launches(1);
  return e;
}

}  // namespace bitlinear
