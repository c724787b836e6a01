// Decode contraction (few tokens, M <= kDecodeMaxM) on the 5th-generation
// tensor cores: y = dequant(x_q . W_q^T) with tcgen05.mma kind::f8f6f4, exact
// in fp32, streaming the 2-bit packed weights from HBM once.
//
// Page "BitNet b1.58 in Production: 1-Bit LLMs and Energy Benchmarks", section
// "The Mathematical Mechanism", items 3-4 (integer accumulation of the ternary
// products, dequantization by gamma * max|x| / Q_b); page "BitNet 1-bit LLM
// Inference Framework", section "How the LUT Kernel Works" (2-bit code
// 00 = 0, 01 = +1, 10 = -1, four weights per byte, int32 accumulation).
//
// Work split.  A CTA owns 128 weight rows (the MMA's M) and a slice of the
// 512-wide K segments.  The S CTAs of a thread-block cluster take the S slices
// of the same 128 rows (split-K); their int32 partial sums meet in the shared
// memory of cluster rank 0 (red.shared::cluster), which dequantizes and
// stores.  The host picks S so that about two CTAs per SM cover the matrix in
// as few segment-times as possible (decode_plan below).
//
// Both operand planes of every token sit in the MMA's n dimension (act_ops.cuh,
// decode layout): columns [0, Mt) accumulate W . (16 h'), [Mt, 2 Mt) W . l', so
// one m128 x n(2 Mt) x k32 MMA covers both, and the exact integer sum of a row
// and token is D[m] + D[Mt + m].  Each column stays below 2^24 in magnitude
// (|W . 16 h'| <= 128 K <= 2^23 for K <= 65536), so the fp32 accumulation is exact.
//
// Roles (192 threads):
//   warp 0      producer: per stage (G segments), one bulk copy of the tile's
//               G segments (contiguous in the tile-major packed layout, up to
//               32 KB: the copy engine's rate per SM grows with the request
//               size) and one bulk copy of the stage's activation blocks
//               (contiguous in the decode layout), each on its own mbarrier.
//               The weight copies of the first NS stages are issued before the
//               wait for the previous kernel, and the decoders start on them.
//   warp 1      allocates 256 TMEM columns (A slots at 0, 64, 128; D at 192),
//               and issues 8 MMAs per half segment (256 k) and commits: the
//               whole warp runs the loop and one elected lane issues (at
//               n = 2 Mt <= 64 an MMA costs the issuing loop, not the tensor
//               pipe: a one-lane loop took about three times as long).
//   warps 2-5   decoders, thread = weight row: 2-bit codes -> e4m3 bytes by
//               byte permutes (kCodeToE4M3), 64 TMEM columns per half segment
//               (tcgen05.st), three A slots in rotation; afterwards the same
//               warps are the epilogue (tcgen05.ld of D, planes combined in
//               int32, split-K reduction, y = fl(fl(acc * act_scale[m]) *
//               w_scale[n])).
// A row's codes are decoded word by word (16 codes): the four TMEM columns of a
// word hold the weights of inputs (0,2,4,6), (8..14 even), (1,3,5,7), (9..15
// odd); the decode operand layout stores the activations in that order.
//
// Shared memory stays between 76 and 113 KB per CTA for Mt <= 24, so exactly
// two CTAs fit on an SM (2 x 256 TMEM columns); Mt = 32 takes one per SM.
//
// Every mbarrier wait is bounded and warp-uniform: on expiry the kernel records
// BITLINEAR_ERR_TIMEOUT, all roles stop, copies and MMAs in flight are waited
// for (bounded), every CTA still meets its cluster peers at the final barrier,
// and TMEM is freed before the CTA exits.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "act_ops.cuh"
#include "device_util.cuh"
#include "internal.h"

namespace bitlinear {
namespace {

constexpr int kRows = 128;                  // weight rows per CTA (MMA M)
constexpr int kThreads = 192;
constexpr uint32_t kTmemCols = 256;
constexpr int kASlots = 3;                  // A slots of 64 columns (256 k)
constexpr uint32_t kColD = 192;             // accumulators: 2 Mt <= 64 columns
constexpr int kMaxStages = 8;
constexpr int kMaxSplit = 8;                // portable cluster size
constexpr uint32_t kSpin = 1u << 24;
constexpr uint32_t kCodeToE4M3 = 0x00B83800u;  // bytes 0x00 (code 0), 0x38 (+1), 0xB8 (-1)
constexpr int kWStageBytes = 128 * 128;     // per segment: 128 rows x 128 bytes of packed codes
constexpr int64_t kTwoPerSm = 115712;       // 2 x (this + 1 KB reserved) = 228 KB per SM
constexpr int64_t kThreePerSm = 76800;      // above this, a third CTA does not fit

struct DecodeTcParams {
  const uint8_t* packed;
  const uint8_t* x_ops;
  const float* act_scale;
  const float* w_scale;
  void* y;
  int32_t* acc_debug;
  int* dev_err;
  const uint8_t* pf;         // L2 prefetch of the caller (or null)
  uint64_t pf_bytes;
  int M, N, out_dtype;
  int nseg, ntiles16;
  int S, G, NS, stage_bytes;
};

// Shared-memory bytes past the stages: split-K partial sums [Mt][128] int32,
// then the mbarriers, the TMEM base and the abort flag.
__host__ __device__ constexpr int red_bytes(int Mt) { return kRows * Mt * 4; }
constexpr int kBarBytes = 8 * (3 * kMaxStages + 2 * kASlots + 2) + 16;

// Bounded wait taken by every lane of a warp with one outcome for all of them:
// the tcgen05 loads and stores that follow are warp-collective.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag, int* dev_err) {
  bool ok = mbar_wait_bounded(bar, parity, kSpin);
  ok = __all_sync(0xffffffffu, ok);
  if (!ok) {
    if ((threadIdx.x & 31) == 0) {
      atomicCAS(dev_err, 0, kDevErrTimeout);
      *abort_flag = 1;
    }
    __syncwarp();
  }
  return ok;
}

// Single-thread version (producer and MMA lanes).
__device__ __forceinline__ bool lane_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag, int* dev_err) {
  if (mbar_wait_bounded(bar, parity, kSpin)) return true;
  atomicCAS(dev_err, 0, kDevErrTimeout);
  *abort_flag = 1;
  return false;
}

__device__ __forceinline__ bool warp_aborted(volatile int* abort_flag) {
  return __any_sync(0xffffffffu, *abort_flag != 0);
}

template <int MT8>
__global__ void __launch_bounds__(kThreads, 1) decode_tc_kernel(const DecodeTcParams p) {
  constexpr int Mt = 8 * MT8;               // tokens padded to 8
  constexpr int Nmma = 2 * Mt;              // MMA n: both planes
  constexpr int kXBlock = 256 * Mt;         // operand bytes per 128 k
  constexpr int kXSeg = 4 * kXBlock;        // operand bytes per 512 k
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  const uint32_t sbase = smem_u32(smem);
  const int off_red = p.NS * p.stage_bytes;
  int* s_red = reinterpret_cast<int*>(smem + off_red);
  const uint32_t full0 = sbase + off_red + red_bytes(Mt);    // weights of a stage landed
  const uint32_t fullx0 = full0 + 8 * kMaxStages;              // operands of a stage landed
  const uint32_t empty0 = fullx0 + 8 * kMaxStages;
  const uint32_t afull0 = empty0 + 8 * kMaxStages;
  const uint32_t aempty0 = afull0 + 8 * kASlots;
  const uint32_t dfull = aempty0 + 8 * kASlots;
  const uint32_t fin = dfull + 8;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + off_red + red_bytes(Mt) + kBarBytes - 16);
  volatile int* s_abort = reinterpret_cast<volatile int*>(s_tmem + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = p.S;
  const int rank = S > 1 ? (int)cluster_ctarank() : 0;
  const int tile = blockIdx.x / S;
  const int s0 = (int)((int64_t)rank * p.nseg / S), s1 = (int)((int64_t)(rank + 1) * p.nseg / S);
  const int nst = (s1 - s0 + p.G - 1) / p.G;                 // stages of this CTA (>= 1)
  const int rows = 16 * min(8, p.ntiles16 - tile * 8);       // weight rows of this tile (<= 128)

  if (threadIdx.x == 0) {
    for (int s = 0; s < p.NS; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(fullx0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 5);          // four decoder warps + one MMA commit
    }
    for (int a = 0; a < kASlots; ++a) {
      mbar_init(afull0 + 8 * a, 4);
      mbar_init(aempty0 + 8 * a, 1);
    }
    mbar_init(dfull, 1);
    mbar_init(fin, 1);
    *s_abort = 0;
    fence_mbar_init();
  }
  if (S > 1 && rank == 0)
    for (int e = threadIdx.x; e < kRows * Mt; e += kThreads) s_red[e] = 0;
  if (warp == 1) tmem_alloc(smem_u32(s_tmem), kTmemCols);
  tc_fence_before();
  __syncthreads();
  if (S > 1) cluster_sync();                 // rank 0's partial-sum buffer is zero before any peer adds
  tc_fence_after();
  pdl_launch_dependents();
  const uint32_t tmem = *s_tmem;

  int acc[Mt];                               // epilogue warps: this row's sums per token
  float as_reg[Mt];                          // per-token scales
  float res_reg[Mt];                         // residual inputs (out_dtype 2)
  float wsn_reg = 0.0f;                      // this row's weight scale
  bool have = false;
  const int r = 32 * (warp & 3) + lane;      // decoder / epilogue row within the tile

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      const uint32_t xoff = (uint32_t)(kWStageBytes * p.G);
      bool waited = false;
      int deferred = 0;                      // stages whose operand copy waits for the previous kernel
      auto issue_x = [&](int st) {
        const int sg = s0 + st * p.G, gc = min(p.G, s1 - sg);
        const int slot = st % p.NS;
        mbar_arrive_expect_tx(fullx0 + 8 * slot, (uint32_t)(gc * kXSeg));
        bulk_g2s(sbase + slot * p.stage_bytes + xoff, p.x_ops + (int64_t)sg * kXSeg, (uint32_t)(gc * kXSeg),
                 fullx0 + 8 * slot);
      };
      int st = 0;
      for (; st < nst; ++st) {
        const int slot = st % p.NS, round = st / p.NS;
        if (round >= 1) {
          if (!waited) {
            l2_prefetch_share(p.pf, p.pf_bytes, 0, 1);   // after this CTA's first weight copies
            pdl_wait();
            waited = true;
            for (int d = st - deferred; d < st; ++d) issue_x(d);
            deferred = 0;
          }
          if (!lane_wait(empty0 + 8 * slot, (round - 1) & 1, s_abort, p.dev_err)) break;
        }
        const int sg = s0 + st * p.G, gc = min(p.G, s1 - sg);
        // segments [sg, sg + gc) of the tile: one contiguous range of the packed layout
        mbar_arrive_expect_tx(full0 + 8 * slot, (uint32_t)(gc * rows * 128));
        bulk_g2s_hint(sbase + slot * p.stage_bytes,
                      p.packed + (int64_t)tile * p.nseg * 16384 + (int64_t)sg * rows * 128,
                      (uint32_t)(gc * rows * 128), full0 + 8 * slot, pol);
        if (waited) issue_x(st);
        else ++deferred;
      }
      if (!waited) {
        l2_prefetch_share(p.pf, p.pf_bytes, 0, 1);
        pdl_wait();
        for (int d = st - deferred; d < st; ++d) issue_x(d);
      }
      // nothing may still be landing in shared memory when the CTA exits
      const int used = st < p.NS ? st : p.NS;
      for (int s = 0; s < used; ++s) {
        const int last = st - 1 - ((st - 1 - s) % p.NS);
        if (!mbar_wait_bounded(full0 + 8 * s, (last / p.NS) & 1, kSpin)) atomicCAS(p.dev_err, 0, kDevErrTimeout);
        if (!mbar_wait_bounded(fullx0 + 8 * s, (last / p.NS) & 1, kSpin)) atomicCAS(p.dev_err, 0, kDevErrTimeout);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issue
    // The whole warp runs the loop (its waits and descriptors are warp-uniform);
    // one elected lane, the same throughout, issues every MMA and commit.
    const uint32_t idesc = idesc_e4m3_f32(kRows, Nmma);
    int a = 0;
    bool first = true, ok = true;
    for (int st = 0; st < nst && ok && !warp_aborted(s_abort); ++st) {
      const int slot = st % p.NS;
      if (!warp_wait(fullx0 + 8 * slot, (st / p.NS) & 1, s_abort, p.dev_err)) break;
      const int sg = s0 + st * p.G, gc = min(p.G, s1 - sg);
      const uint32_t xs = sbase + slot * p.stage_bytes + (uint32_t)(kWStageBytes * p.G);
      for (int g = 0; g < gc && ok; ++g) {
        for (int h = 0; h < 2; ++h) {
          const int as = a % kASlots;
          if (!warp_wait(afull0 + 8 * as, (a / kASlots) & 1, s_abort, p.dev_err)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int s = 0; s < 8; ++s) {      // k32 steps of this half segment
            const uint32_t b = xs + g * kXSeg + (2 * h + (s >> 2)) * kXBlock + 32 * (s & 3);
            if (elect_one())
              mma_f8f6f4_ts(tmem + kColD, tmem + as * 64 + 8 * s, smem_desc_sw128(b), idesc, first ? 0u : 1u);
            __syncwarp();
            first = false;
          }
          if (elect_one()) mma_commit(aempty0 + 8 * as);    // the A slot may be rewritten
          __syncwarp();
          ++a;
        }
      }
      if (ok) {
        if (elect_one()) mma_commit(empty0 + 8 * slot);     // the stage's operands are read
        __syncwarp();
      }
    }
    if (elect_one()) {
      mma_commit(dfull);                     // accumulators complete
      mma_commit(fin);                       // before TMEM is freed every MMA issued here must be finished
    }
    __syncwarp();
    if (lane == 0 && !mbar_wait_bounded(fin, 0, kSpin)) atomicCAS(p.dev_err, 0, kDevErrTimeout);
    __syncwarp();
  } else {
    // ------------------------------------------------------------ decoders
    const uint32_t lane_addr = (uint32_t)(32 * (warp & 3)) << 16;
    const bool valid = r < rows;
    int a = 0;
    bool ok = true;
    for (int st = 0; st < nst && ok && !warp_aborted(s_abort); ++st) {
      const int slot = st % p.NS;
      if (!warp_wait(full0 + 8 * slot, (st / p.NS) & 1, s_abort, p.dev_err)) break;
      const int sg = s0 + st * p.G, gc = min(p.G, s1 - sg);
      // segment g of the stage: rows x 128 bytes; row r at line r, chunk c stored at c ^ (r % 8)
      const uint32_t wrow = sbase + slot * p.stage_bytes + r * 128;
      for (int g = 0; g < gc && ok; ++g) {
        for (int h = 0; h < 2; ++h) {
          const int as = a % kASlots;
          if (a >= kASlots && !warp_wait(aempty0 + 8 * as, ((a / kASlots) - 1) & 1, s_abort, p.dev_err)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int cp = 0; cp < 2; ++cp) {   // 32 TMEM columns = two 16-byte chunks
            uint32_t cols[32];
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
              const int c = 4 * h + 2 * cp + cc;
              const uint4 v = valid ? lds128(wrow + g * rows * 128 + (uint32_t)((c ^ (r & 7)) << 4))
                                    : make_uint4(0u, 0u, 0u, 0u);
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
            tmem_st32(tmem + lane_addr + as * 64 + cp * 32, cols);
          }
          tmem_wait_st();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(afull0 + 8 * as);        // A slot written
          ++a;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty0 + 8 * slot);          // weight stage read
    }

    // ------------------------------------------------------------ epilogue
    pdl_wait();                              // act_scale and y follow the stream order
    // The scales are loaded now, while the MMAs finish: in the store loop below
    // the compiler could not move them above the (possibly aliasing) y stores.
#pragma unroll
    for (int m = 0; m < Mt; ++m) as_reg[m] = m < p.M ? __ldcg(p.act_scale + m) : 0.0f;
    wsn_reg = (tile * kRows + r < p.N) ? __ldg(p.w_scale + tile * kRows + r) : 0.0f;
    if (p.out_dtype == 2 && rank == 0 && tile * kRows + r < p.N) {   // the residuals, for the same reason
      const unsigned short* yr = reinterpret_cast<const unsigned short*>(p.y) + tile * kRows + r;
#pragma unroll
      for (int m = 0; m < Mt; ++m)
        res_reg[m] = m < p.M ? __uint_as_float((uint32_t)__ldcg(yr + (size_t)m * p.N) << 16) : 0.0f;
    }
    if (!warp_aborted(s_abort) && warp_wait(dfull, 0, s_abort, p.dev_err)) {
      tc_fence_after();
      uint32_t d[Nmma];
#pragma unroll
      for (int c = 0; c < Nmma / 8; ++c) {
        uint32_t v8[8];
        tmem_ld8(tmem + lane_addr + kColD + 8 * c, v8);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 8; ++j) d[8 * c + j] = v8[j];
      }
#pragma unroll
      for (int m = 0; m < Mt; ++m)
        acc[m] = (int)__uint_as_float(d[m]) + (int)__uint_as_float(d[Mt + m]);
      have = true;
      if (S > 1 && rank != 0 && valid) {
        const uint32_t red0 = map_shared_rank(smem_u32(s_red), 0);
#pragma unroll
        for (int m = 0; m < Mt; ++m)
          if (m < p.M) red_add_shared_cluster(red0 + (uint32_t)(m * kRows + r) * 4, acc[m]);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (S > 1) cluster_sync();                 // every peer's partial sums are in rank 0
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);

  if (warp >= 2 && have && rank == 0) {
    const int n = tile * kRows + r;
    if (n < p.N && !*s_abort) {
      const float wsn = wsn_reg;
#pragma unroll
      for (int m = 0; m < Mt; ++m) {
        if (m < p.M) {
          const int v = S > 1 ? acc[m] + s_red[m * kRows + r] : acc[m];
          const float as = as_reg[m];
          const size_t o = (size_t)m * p.N + n;
          const float yv = __fmul_rn(__fmul_rn((float)v, as), wsn);
          if (p.out_dtype == 0) {
            reinterpret_cast<float*>(p.y)[o] = yv;
          } else {
            __nv_bfloat16* yb = reinterpret_cast<__nv_bfloat16*>(p.y) + o;
            // out_dtype 2: residual add into the bf16 output, y = bf16(y + result)
            *yb = __float2bfloat16_rn(p.out_dtype == 2 ? __fadd_rn(res_reg[m], yv) : yv);
          }
          if (p.acc_debug) p.acc_debug[o] = v;
        }
      }
    }
  }
}

// x_q -> activation operands, for callers that did not get them from quant_act.
__global__ void act_ops_from_codes_kernel(const int8_t* __restrict__ x_q, int64_t M, int64_t K,
                                          int64_t Kp, uint8_t* __restrict__ ops) {
  pdl_launch_dependents();                   // the next kernel waits for this one to complete
  pdl_wait();
  const int64_t per_row = Kp >> 4;
  for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < M * per_row;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int64_t m = idx / per_row, k = (idx - m * per_row) << 4;
    uint32_t q[4];
#pragma unroll
    for (int hv = 0; hv < 2; ++hv) {
      const uint2 v = k + 8 * hv < K ? *reinterpret_cast<const uint2*>(x_q + m * K + k + 8 * hv) : make_uint2(0u, 0u);
      q[2 * hv] = v.x;
      q[2 * hv + 1] = v.y;
    }
    write_act_ops16_any(ops, M, m, k, Kp, q);
  }
}

}  // namespace

// Split-K and staging plan of a decode launch.
DecodePlan decode_plan(int64_t M, int64_t N, int64_t K, int sms) {
  DecodePlan pl = {};
  const int Mt = (int)act_ops_mt(M);
  pl.Mt = Mt;
  pl.nseg = (int)(act_ops_kpad(K) / 512);
  pl.ntile = (int)((N + kRows - 1) / kRows);
  const int64_t fixed = 1024 + red_bytes(Mt) + kBarBytes;
  const int64_t seg_bytes = kWStageBytes + 4 * 256 * Mt;   // weights + operands of one segment
  // two segments per stage (32 KB weight copies) when two such stages fit twice per SM
  pl.G = fixed + 4 * seg_bytes <= kTwoPerSm ? 2 : 1;
  pl.stage_bytes = (int)(pl.G * seg_bytes);
  int NS = 2;
  while (NS < kMaxStages && fixed + (int64_t)(NS + 1) * pl.stage_bytes <= kTwoPerSm) ++NS;
  pl.NS = NS;
  pl.smem = fixed + (int64_t)NS * pl.stage_bytes;
  const int per_sm = pl.smem <= kTwoPerSm ? 2 : 1;
  const int64_t slots = (int64_t)per_sm * sms;
  // S: fewest segment-times, counting one segment of fixed cost per CTA and
  // whole waves of `slots` CTAs; ties go to the smaller S.  A split leaves each
  // CTA at least two segments: a cluster starts only when all of its CTAs find
  // room in one GPC, which in a chain of launches overlapping by programmatic
  // dependent launch delayed whole clusters by several microseconds, and with
  // one segment per CTA that delay is not amortized (8B O projection, 16 tokens:
  // 10.4 us in clusters of 8, 7.0 us in clusters of 4).
  // From 16 tokens a grid that puts two CTAs on some SMs costs 2.5 segments more
  // (measured: 8B QKV at 16 tokens 8.2 us in 96 CTAs of four segments, 8.9 us in
  // 192 CTAs of two; at 4 tokens the 192 CTAs win).  Costs in half segments.
  const int64_t crowd = Mt >= 16 ? 5 : 0;
  int64_t best = -1;
  pl.S = 1;
  for (int S = 1; S <= kMaxSplit && S <= pl.nseg; ++S) {
    if (S > 1 && (pl.nseg + S - 1) / S < 2) break;
    const int64_t ctas = (int64_t)pl.ntile * S;
    const int64_t waves = (ctas + slots - 1) / slots;
    const int64_t cost = 2 * waves * ((pl.nseg + S - 1) / S + 1) + (ctas > sms ? crowd : 0);
    if (best < 0 || cost < best) {
      best = cost;
      pl.S = S;
    }
  }
  return pl;
}

bool decode_plan_ok(const DecodePlan& pl) {
  return pl.smem > kThreePerSm && pl.smem <= 227 * 1024 && pl.NS >= 2 && pl.NS <= kMaxStages &&
         pl.S >= 1 && pl.S <= kMaxSplit && pl.S <= pl.nseg && pl.Mt % 8 == 0 && pl.Mt >= 8 &&
         pl.Mt <= kDecodeMaxM && 2 * pl.Mt + (int)kColD <= (int)kTmemCols;
}

size_t act_ops_bytes(int64_t M, int64_t K) {
  return (size_t)(2 * (act_ops_prefill(M) ? act_ops_mpad(M) : act_ops_mt(M)) * act_ops_kpad(K));
}

cudaError_t launch_act_ops_from_codes(const int8_t* x_q, int64_t M, int64_t K, uint8_t* ops,
                                      bool pdl, cudaStream_t stream) {
  const int64_t Kp = act_ops_kpad(K);
  const int64_t work = M * (Kp >> 4);
  int64_t blocks = (work + 255) / 256;
  if (blocks > (int64_t)num_sms() * 8) blocks = (int64_t)num_sms() * 8;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks, 1, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  cudaError_t e = cudaLaunchKernelEx(&cfg, act_ops_from_codes_kernel, x_q, M, K, Kp, ops);
  count_launches(1);
  return e;
}

cudaError_t launch_decode_tc(const uint8_t* x_ops, const float* act_scale, const uint8_t* packed,
                             const float* w_scale, int64_t M, int64_t N, int64_t K, int out_dtype,
                             void* y, int32_t* acc_debug, int* dev_err, bool pdl,
                             cudaStream_t stream, L2Prefetch pf) {
  const DecodePlan pl = decode_plan(M, N, K, num_sms());
  if (!decode_plan_ok(pl)) return cudaErrorInvalidValue;
  DecodeTcParams p = {};
  p.packed = packed;
  p.x_ops = x_ops;
  p.act_scale = act_scale;
  p.w_scale = w_scale;
  p.y = y;
  p.acc_debug = acc_debug;
  p.dev_err = dev_err;
  p.pf = pf.p;
  p.pf_bytes = pf.bytes;
  p.M = (int)M;
  p.N = (int)N;
  p.out_dtype = out_dtype;
  p.nseg = pl.nseg;
  p.ntiles16 = (int)(N / 16);
  p.S = pl.S;
  p.G = pl.G;
  p.NS = pl.NS;
  p.stage_bytes = pl.stage_bytes;
  static bool attr_set = false;
  if (!attr_set) {
    for (void* f : {(void*)decode_tc_kernel<1>, (void*)decode_tc_kernel<2>, (void*)decode_tc_kernel<3>,
                    (void*)decode_tc_kernel<4>}) {
      cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
      if (e != cudaSuccess) return e;
    }
    attr_set = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(pl.ntile * pl.S), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = (size_t)pl.smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  int na = 0;
  attr[na].id = cudaLaunchAttributeClusterDimension;
  attr[na].val.clusterDim.x = (unsigned)pl.S;
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
  switch (pl.Mt / 8) {
    case 1: e = cudaLaunchKernelEx(&cfg, decode_tc_kernel<1>, p); break;
    case 2: e = cudaLaunchKernelEx(&cfg, decode_tc_kernel<2>, p); break;
    case 3: e = cudaLaunchKernelEx(&cfg, decode_tc_kernel<3>, p); break;
    default: e = cudaLaunchKernelEx(&cfg, decode_tc_kernel<4>, p); break;
  }
  count_launches(1);
  return e;
}

}  // namespace bitlinear
