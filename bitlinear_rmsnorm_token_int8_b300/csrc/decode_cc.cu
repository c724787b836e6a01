// Decode contraction for one or two tokens on the CUDA cores, as a
// persistent kernel: y = dequant(x_q . W_q^T) from the int8 codes, or the whole
// BitLinear layer (RMSNorm + absmax quantization of the tokens, then the
// contraction) in one launch.
//
// Page "BitNet b1.58 in Production: 1-Bit LLMs and Energy Benchmarks", section
// "The Mathematical Mechanism", items 2-4 (per-token absmax codes, integer
// product, rescale by the two scales) and bit_linear.py BitLinear.forward
// (RMSNorm, then activation_quant); page "BitNet 1-bit LLM Inference
// Framework", section "How the LUT Kernel Works" (the 2-bit code, integer
// accumulation of the ternary products).
//
// Why persistent: in a chain of dependent decode launches a kernel that
// re-did its setup in every one of thousands of small CTAs (a second wave
// restarting its loads after the first, the row statistics recomputed per
// CTA) was bound by instructions and latency, not by its weight stream.  Here
// one CTA of 512 threads runs per SM and does that work once.
//
// Work split.  A row is read by 8 KS lanes (KS = 1, 2 or 4): lane (ks, c)
// takes the 16-byte chunk c (64 inputs) of segments ks, ks + KS, ... of the
// tile-major packed layout, so a warp covers a group of 4 / KS rows.  The
// groups are split evenly over the CTAs; the 16 warps of a CTA take its groups
// in turn.  A lane's chunks of a row form items of up to kCB chunks.
//
// Weights travel global -> shared memory by 16-byte cp.async into a
// lane-private ring of S items (S = 2 or 3), so a warp keeps up to
// S x 32 x kCB x 16 bytes in flight without holding registers; the first S
// items are requested before the wait for the previous kernel (the packed
// weights are not written by in-flight work).  Each lane reads back only the
// chunks it copied itself, so its own cp.async.wait_group orders them.
//
// Activations.  After the wait the CTA stages the tokens' int8 codes in
// shared memory, permuted per 16 inputs like the expanded weight words
// (80-byte pitch per 64-byte chunk: the eight chunk readers of a warp hit
// distinct banks).  Given x_q they are copied; in the layer form every CTA
// quantizes the tokens itself with the thread-to-input mapping, per-thread
// order and reduction tree of quant_act_kernel (thread u takes inputs
// 16u..16u+15; the tree spans that kernel's warps, the others add nothing),
// so codes and scales equal the separate quantization bit for bit.  Rows of
// more than 512 units (that kernel runs up to 1024 threads on them) take the
// variant in which each thread plays two of its threads.  Its token
// row arrives by one bulk copy into shared memory, through the copy engine
// rather than behind the ring's first S items of 16-byte requests (8B gate+up
// at one token: 12.8 -> 12.5-12.6 us per launch).
//
// A 32-bit word of codes (16 inputs) is expanded by byte permutes into int8
// words of inputs (0,2,4,6), (8..14 even), (1,3,5,7), (9..15 odd) (code
// 0 -> 0, 1 -> +1, 2 -> -1); a word is four dp4a per token.  The int32 sums
// are exact (|acc| <= 128 K < 2^31).  At a group's last item the row's lanes
// reduce with shuffles and lane (ks = 0, c = m) writes token m:
// y = fl(fl(acc * sigma_m) * w_scale[n]).
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "act_ops.cuh"
#include "device_util.cuh"
#include "internal.h"
#include "quant_math.cuh"

namespace bitlinear {
namespace {

constexpr int kCcThreads = 512;                // 16 warps
constexpr int kCcWarps = kCcThreads / 32;
constexpr int kCB = 8;                         // chunks per lane per item
constexpr int kItemBytes = 32 * kCB * 16;      // one warp's item: 4 KB
constexpr int kChunkPitch = 80;                // a staged 64-byte chunk + 16 bytes
constexpr int kSegPitch = 8 * kChunkPitch;     // one token's 512 inputs in shared memory
constexpr uint32_t kCodeToI8 = 0x00FF0100u;    // bytes 0x00 (code 0), 0x01 (+1), 0xFF (-1)
constexpr int kFusedMaxK = 16384;              // layer form: quant_act_kernel's threads <= 1024
constexpr int64_t kSmemCap = 220 * 1024;       // dynamic shared memory budget per CTA
constexpr uint32_t kSpin = 1u << 24;           // polls of a bounded mbarrier wait

struct DecodeCcParams {
  const uint8_t* packed;
  const float* w_scale;
  void* y;
  int32_t* acc_debug;
  const uint8_t* pf;         // L2 prefetch of the caller (or null)
  uint64_t pf_bytes;
  // codes form
  const int8_t* x_q;
  const float* act_scale;
  // layer form
  const uint4* x;            // bf16 rows, 8 per vector
  const uint4* gain;         // bf16 [K] or null
  float rms_eps;
  int8_t* x_q_out;           // [M, K] out, or null
  float* act_scale_out;      // [M] out, or null
  int* dev_err;              // layer form: error word (a copy that never landed)
  int M, N, K, nseg, Np, out_dtype;
  int ngroups;               // Np * KS / 4
  int nb;                    // items per row group
  int S;                     // ring stages (2 or 3)
  int Tq;                    // quant_act_kernel's threads for one row (layer form)
};

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint64_t policy) {
  asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "l"(policy)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// 16 inputs of one token in natural order (x = [0..3], y = [4..7], z = [8..11],
// w = [12..15]) rearranged like the expanded weight words.
__device__ __forceinline__ uint4 permute16(uint4 v) {
  return make_uint4(__byte_perm(v.x, v.y, 0x6420), __byte_perm(v.z, v.w, 0x6420), __byte_perm(v.x, v.y, 0x7531),
                    __byte_perm(v.z, v.w, 0x7531));
}

// acc[m] += the 64 products of one 16-byte chunk of codes with token m's staged
// inputs at shared address xs + m * tstride.
template <int MT>
__device__ __forceinline__ void dot_chunk(const uint4 w, uint32_t xs, uint32_t tstride, int (&acc)[MT]) {
  const uint32_t wd[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t lo = wd[j] & 0x33333333u, hi = (wd[j] >> 2) & 0x33333333u;
    const int w0 = (int)__byte_perm(kCodeToI8, 0u, lo);          // inputs 0, 2, 4, 6
    const int w1 = (int)__byte_perm(kCodeToI8, 0u, lo >> 16);    // 8, 10, 12, 14
    const int w2 = (int)__byte_perm(kCodeToI8, 0u, hi);          // 1, 3, 5, 7
    const int w3 = (int)__byte_perm(kCodeToI8, 0u, hi >> 16);    // 9, 11, 13, 15
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      const uint4 xv = lds128(xs + m * tstride + 16 * j);
      acc[m] = __dp4a(w0, (int)xv.x, acc[m]);
      acc[m] = __dp4a(w1, (int)xv.y, acc[m]);
      acc[m] = __dp4a(w2, (int)xv.z, acc[m]);
      acc[m] = __dp4a(w3, (int)xv.w, acc[m]);
    }
  }
}

// MT: tokens the kernel is compiled for (M <= MT).  KS: lanes per (row, chunk).
// FUSED: the layer form (quantize x) instead of reading x_q.
// FUSED: 0 for the codes form; 1 or 2 for the layer form, the number of
// quant_act_kernel threads each thread plays (2 for rows of more than 512 units).
template <int MT, int KS, int FUSED>
__global__ void __launch_bounds__(kCcThreads, 1) decode_cc_kernel(const DecodeCcParams p) {
  extern __shared__ __align__(16) uint8_t dsm[];
  __shared__ float s_max[MT][32];
  __shared__ float2 s_ss[MT][32];
  __shared__ float s_m[MT], s_sum[MT], s_sigma[MT];
  __shared__ __align__(8) uint64_t s_xbar;       // layer form: the token row's bulk copy
  constexpr int kRowsPerWarp = 4 / KS;
  constexpr int kLog2KS = KS == 1 ? 0 : KS == 2 ? 1 : 2;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int c = lane & 7;                                        // chunk of a segment
  const int ks = (lane >> 3) & (KS - 1);                         // first segment of this lane
  const int lrow = lane >> (3 + kLog2KS);                        // row within the group
  const int S = p.S;
  const uint32_t ring = smem_u32(dsm) + (uint32_t)(warp * S * kItemBytes) + (uint32_t)(lane * 16);
  uint8_t* const xst = dsm + (size_t)kCcWarps * S * kItemBytes;  // the tokens' staged codes
  const uint32_t xsm = smem_u32(xst);
  const uint32_t tstride = (uint32_t)(p.nseg * kSegPitch);

  // this CTA's row groups, and this warp's share of them (groups g0 + warp + 16 j)
  const int g0 = (int)((int64_t)blockIdx.x * p.ngroups / gridDim.x);
  const int g1 = (int)((int64_t)(blockIdx.x + 1) * p.ngroups / gridDim.x);
  const int ngw = g1 - g0 > warp ? (g1 - g0 - warp + kCcWarps - 1) / kCcWarps : 0;
  const uint64_t pol = policy_evict_first();

  // The issue cursor walks this warp's items in order: group ij (rows of group
  // g0 + warp + 16 ij), chunk batch ib = chunks [ib kCB, (ib + 1) kCB) of the lane's
  // row, into ring slot islot.  iw: the lane's chunk of its row in the cursor's group
  // at segment ks; istep: bytes between consecutive segments of that row (R x 128 in
  // a tile of R rows).
  int ij = 0, ib = 0, islot = 0, istep = 0;
  const uint8_t* iw = nullptr;
  auto issue = [&]() {
    if (ij < ngw) {
      if (ib == 0) {
        const int row = (g0 + warp + kCcWarps * ij) * kRowsPerWarp + lrow;   // < Np
        const int tile = row >> 7, r = row & 127;
        istep = min(128, p.Np - tile * 128) * 128;
        iw = p.packed + (size_t)tile * p.nseg * 16384 + (size_t)r * 128 + ((c ^ (r & 7)) << 4) + (size_t)ks * istep;
      }
      const uint32_t slot = ring + (uint32_t)(islot * kItemBytes);
      const uint8_t* src = iw + (size_t)(ib * kCB * KS) * istep;
#pragma unroll
      for (int i = 0; i < kCB; ++i)
        if (ks + KS * (ib * kCB + i) < p.nseg) cp_async16(slot + i * 512, src + (size_t)(i * KS) * istep, pol);
      if (++ib == p.nb) {
        ib = 0;
        ++ij;
      }
    }
    cp_async_commit();                       // one group per item, empty past the end
    islot = islot + 1 == S ? 0 : islot + 1;
  };

  const uint32_t xbar = smem_u32(&s_xbar);
  if constexpr (FUSED) {
    if (tid == 0) {
      mbar_init(xbar, 1);
      fence_mbar_init();
    }
    __syncthreads();
  }

  for (int n = 0; n < S; ++n) issue();       // weights: before the wait

  // the layer form's RMSNorm gain (not written by earlier kernels) of the units
  // tid and tid + kCcThreads (quant_act_kernel's threads tid and tid + 512)
  constexpr int kVT = FUSED > 1 ? 2 : 1;
  uint4 gv[kVT][2];
  const int V = p.K >> 3, U = (V + 1) >> 1;
  if constexpr (FUSED) {
#pragma unroll
    for (int vt = 0; vt < kVT; ++vt)
#pragma unroll
      for (int hv = 0; hv < 2; ++hv) {
        const int u = tid + vt * kCcThreads, v = 2 * u + hv;
        gv[vt][hv] = (p.gain && u < U && v < V) ? __ldg(p.gain + v) : kOnes;
      }
  }
  if (warp == 0) l2_prefetch_share(p.pf, p.pf_bytes, lane, 32);
  pdl_launch_dependents();
  pdl_wait();                                // x, x_q, act_scale and y follow the stream order

  // ---- the tokens' codes into shared memory
  bool x_landed = true;
  if constexpr (FUSED) {
    // The token row (M = 1) comes in as one bulk copy: through the copy engine it
    // does not queue behind the weight ring's cp.async requests issued above.
    const uint32_t xrow = xsm + MT * tstride;
    if (tid == 0) {
      mbar_arrive_expect_tx(xbar, (uint32_t)p.K * 2u);
      bulk_g2s(xrow, p.x, (uint32_t)p.K * 2u, xbar);
    }
    x_landed = mbar_wait_bounded(xbar, 0, kSpin);
    if (!x_landed) atomicCAS(p.dev_err, 0, kDevErrTimeout);
    // statistics of the token row (M = 1) as quant_act_kernel with p.Tq threads
    // (up to 1024): its thread u < U takes inputs 16u..16u+15 (vectors 2u, 2u + 1),
    // in that order; thread tid here plays its thread tid and, for rows of more
    // than 512 units, its thread tid + 512 (warps warp and warp + 16 there).
    static_assert(!FUSED || MT == 1, "the layer form takes one token");
    constexpr bool two = kVT > 1;
    // unit u's vectors into x, its statistics through that kernel's warp tree into slot
    auto unit_stats = [&](int u, uint4 (&x)[2], const uint4 (&g)[2], int slot) {
      float amax = 0.0f, hi = 0.0f, lo = 0.0f;
#pragma unroll
      for (int hv = 0; hv < 2; ++hv) {
        const int v = 2 * u + hv;
        if (u < U && v < V) {
          x[hv] = lds128(xrow + 16 * v);
          float xf[8], gf[8];
          unpack8(x[hv], xf);
          unpack8(g[hv], gf);
#pragma unroll
          for (int jj = 0; jj < 8; ++jj) {
            amax = fmaxf(amax, fabsf(__fmul_rn(xf[jj], gf[jj])));
            float s_, e_;
            two_sum(hi, __fmul_rn(xf[jj], xf[jj]), s_, e_);   // x^2 is exact in fp32
            hi = s_;
            lo = __fadd_rn(lo, e_);
          }
        } else {
          x[hv] = make_uint4(0u, 0u, 0u, 0u);
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {     // the warp's xor tree, as block_stats
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        const float h2 = __shfl_xor_sync(0xffffffffu, hi, o), l2 = __shfl_xor_sync(0xffffffffu, lo, o);
        pair_add(hi, lo, h2, l2);
      }
      if (lane == 0) {
        s_max[0][slot] = amax;
        s_ss[0][slot] = make_float2(hi, lo);
      }
    };
    uint4 xv0[2], xv1[2];
    unit_stats(tid, xv0, gv[0], warp);
    if constexpr (two) unit_stats(tid + kCcThreads, xv1, gv[kVT - 1], warp + 16);
    __syncthreads();
    // warp 0: the tree over that kernel's p.Tq / 32 warps (zero beyond them)
    const int nwq = p.Tq >> 5;
    if (warp == 0) {
      float a = lane < nwq ? s_max[0][lane] : 0.0f;
      float2 p2 = lane < nwq ? s_ss[0][lane] : make_float2(0.0f, 0.0f);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
        const float h2 = __shfl_xor_sync(0xffffffffu, p2.x, o), l2 = __shfl_xor_sync(0xffffffffu, p2.y, o);
        pair_add(p2.x, p2.y, h2, l2);
      }
      if (lane == 0) {
        s_m[0] = a;
        s_sum[0] = __fadd_rn(p2.x, p2.y);
      }
    }
    __syncthreads();
    // codes of the units (zero past K), staged permuted
    const RowQuant rq = row_quant(s_m[0], s_sum[0], p.K, p.rms_eps);
    if (tid == 0) {
      s_sigma[0] = rq.sigma;
      if (blockIdx.x == 0 && p.act_scale_out) p.act_scale_out[0] = rq.sigma;
    }
    auto unit_codes = [&](int u, const uint4 (&x)[2], const uint4 (&g)[2]) {
      if (u >= p.nseg * 32) return;
      const int sgm = u >> 5, cc = (u >> 2) & 7, jj = u & 3;
      uint32_t w[4];
      row_codes<16>([&](int e) { return __fmul_rn(bf16_at(x[e >> 3], e & 7), bf16_at(g[e >> 3], e & 7)); }, rq, w);
      const uint4 codes = make_uint4(w[0], w[1], w[2], w[3]);
      *reinterpret_cast<uint4*>(xst + sgm * kSegPitch + cc * kChunkPitch + 16 * jj) = permute16(codes);
      if (blockIdx.x == 0 && p.x_q_out && u < U) *reinterpret_cast<uint4*>(p.x_q_out + 16 * u) = codes;
    };
    unit_codes(tid, xv0, gv[0]);
    if constexpr (two) unit_codes(tid + kCcThreads, xv1, gv[kVT - 1]);
  } else {
    const int groupsK = p.nseg * 32;         // 16-input groups per token (Kp / 16)
    for (int i = tid; i < MT * groupsK; i += kCcThreads) {
      const int m = i / groupsK, g = i - m * groupsK;
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (m < p.M && 16 * g < p.K) v = __ldcg(reinterpret_cast<const uint4*>(p.x_q + (size_t)m * p.K) + g);
      const int s = g >> 5, cc = (g >> 2) & 7, jj = g & 3;
      *reinterpret_cast<uint4*>(xst + m * tstride + s * kSegPitch + cc * kChunkPitch + 16 * jj) = permute16(v);
    }
    if (tid < MT) s_sigma[tid] = tid < p.M ? __ldcg(p.act_scale + tid) : 0.0f;
  }
  __syncthreads();

  float sig[MT];
#pragma unroll
  for (int m = 0; m < MT; ++m) sig[m] = s_sigma[m];

  // ---- the weight stream
  int acc[MT];
#pragma unroll
  for (int m = 0; m < MT; ++m) acc[m] = 0;
  const uint32_t xs = xsm + c * kChunkPitch;
  float sc = 0.0f;                           // this lane's token scale (token c)
#pragma unroll
  for (int m = 0; m < MT; ++m)
    if (m == c) sc = sig[m];
  int cslot = 0;                             // ring slot of the item being consumed
  for (int j = 0; j < ngw; ++j) {
    const int row = (g0 + warp + kCcWarps * j) * kRowsPerWarp + lrow;
    const bool out = row < p.N && ks == 0 && c < p.M;       // this lane stores token c of the row
    float wsn = 0.0f, res = 0.0f;
    if (out) {                               // loads whose latency the group's items hide
      wsn = __ldg(p.w_scale + row);
      if (p.out_dtype == 2)
        res = __uint_as_float((uint32_t)__ldcg(reinterpret_cast<const unsigned short*>(p.y) + (size_t)c * p.N + row)
                              << 16);
    }
    for (int b = 0; b < p.nb; ++b) {
      if (S == 3) cp_async_wait<2>();        // this item has landed (the next two may be in flight)
      else cp_async_wait<1>();
      const uint32_t slot = ring + (uint32_t)(cslot * kItemBytes);
#pragma unroll
      for (int i = 0; i < kCB; ++i) {
        const int s = ks + KS * (b * kCB + i);
        if (s < p.nseg) dot_chunk<MT>(lds128(slot + i * 512), xs + s * kSegPitch, tstride, acc);
      }
      issue();                               // refill the slot just read
      cslot = cslot + 1 == S ? 0 : cslot + 1;
    }
    // sum over the row's 8 KS lanes; lane (ks = 0, c) keeps token c
    int mine = 0;
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      int v = acc[m];
#pragma unroll
      for (int o = 1; o < 8 * KS; o <<= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      if (m == c) mine = v;
      acc[m] = 0;
    }
    if (out) {
      const size_t o = (size_t)c * p.N + row;
      const float yv = __fmul_rn(__fmul_rn((float)mine, sc), wsn);
      if (p.out_dtype == 0) reinterpret_cast<float*>(p.y)[o] = yv;
      else if (p.out_dtype == 1) reinterpret_cast<__nv_bfloat16*>(p.y)[o] = __float2bfloat16_rn(yv);
      else reinterpret_cast<__nv_bfloat16*>(p.y)[o] = __float2bfloat16_rn(__fadd_rn(res, yv));
      if (p.acc_debug) p.acc_debug[o] = mine;
    }
  }
  cp_async_wait<0>();                        // nothing may still be landing when the CTA exits
  if (!x_landed) mbar_wait_bounded(xbar, 0, kSpin);
}

// Lanes per (row, chunk): the fewest that still give every warp of the grid a row
// group (fewer lanes per row: longer items, less loop overhead per byte); 4 at most.
int cc_split(int64_t Np, int sms) {
  int ks = 1;
  while (ks < 4 && Np * ks / 4 < (int64_t)sms * kCcWarps) ks *= 2;
  return ks;
}

int64_t cc_staging(int64_t M, int64_t K) {
  const int MT = M <= 1 ? 1 : 2;
  return (int64_t)MT * (act_ops_kpad(K) / 512) * kSegPitch;
}

int cc_stages(int64_t M, int64_t K, int64_t extra = 0) {
  for (int S = 3; S >= 2; --S)
    if ((int64_t)kCcWarps * S * kItemBytes + cc_staging(M, K) + extra <= kSmemCap) return S;
  return 0;
}

template <int MT, int KS, int FUSED>
cudaError_t launch_cfg(const DecodeCcParams& p, int grid, size_t smem, bool pdl, cudaStream_t stream) {
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(decode_cc_kernel<MT, KS, FUSED>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kSmemCap);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid, 1, 1);
  cfg.blockDim = dim3(kCcThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, decode_cc_kernel<MT, KS, FUSED>, p);
}

template <int MT, int FUSED>
cudaError_t launch_mt(const DecodeCcParams& p, int KS, int grid, size_t smem, bool pdl, cudaStream_t stream) {
  if (KS == 4) return launch_cfg<MT, 4, FUSED>(p, grid, smem, pdl, stream);
  if (KS == 2) return launch_cfg<MT, 2, FUSED>(p, grid, smem, pdl, stream);
  return launch_cfg<MT, 1, FUSED>(p, grid, smem, pdl, stream);
}

// Fills the shape fields and launches the kernel for M tokens.
cudaError_t launch_cc(DecodeCcParams& p, int64_t M, int64_t N, int64_t K, bool fused, bool pdl,
                      cudaStream_t stream) {
  const int sms = num_sms();
  p.M = (int)M;
  p.N = (int)N;
  p.K = (int)K;
  p.nseg = (int)(act_ops_kpad(K) / 512);
  p.Np = (int)packed_rows(N);
  const int KS = cc_split(p.Np, sms);
  p.ngroups = p.Np * KS / 4;
  p.nb = ((p.nseg + KS - 1) / KS + kCB - 1) / kCB;
  const int64_t xrow_bytes = fused ? 2 * K : 0;   // the layer form's token row
  p.S = cc_stages(M, K, xrow_bytes);
  p.Tq = (int)((K / 16 + 31) / 32 * 32);
  if (p.S == 0) return cudaErrorInvalidValue;
  const int grid = p.ngroups < sms ? p.ngroups : sms;
  const size_t smem = (size_t)kCcWarps * p.S * kItemBytes + (size_t)cc_staging(M, K) + (size_t)xrow_bytes;
  cudaError_t e;
  if (fused) {
    e = p.Tq > kCcThreads ? launch_mt<1, 2>(p, KS, grid, smem, pdl, stream)
                          : launch_mt<1, 1>(p, KS, grid, smem, pdl, stream);
  } else {
    e = M <= 1 ? launch_mt<1, 0>(p, KS, grid, smem, pdl, stream)
               : launch_mt<2, 0>(p, KS, grid, smem, pdl, stream);
  }
  count_launches(1);
  return e;
}

}  // namespace

// bitlinear_forward given x_q contracts on the codes here for one or two tokens,
// when the staged codes and the weight ring fit in shared memory.  From three
// tokens on the tensor-core kernel wins: its cost per weight (the 2-bit -> e4m3
// expansion) does not grow with the tokens, the dp4a work here does.
bool codes_route(int64_t M, int64_t N, int64_t K) {
  (void)N;
  return M >= 1 && M <= kCodesMaxM && cc_stages(M, K) > 0;
}

// The layer form: one token, whose quant_act_kernel row (up to 1024 threads) this
// kernel's 512 threads can play (K <= 16384).
// Measured in chains of dependent launches: for one token the in-kernel
// quantization costs less than a separate quantization launch; for two it costs
// more (8B gate+up at two tokens: 19.2 us as one kernel, 13.8 + ~3.5 us as two).
bool fused_route(int64_t M, int64_t N, int64_t K) {
  if (!(M == 1 && codes_route(M, N, K) && K <= kFusedMaxK && cc_stages(M, K, 2 * K) > 0)) return false;
  // above 8192 inputs only this persistent kernel has a layer form (the small-CTA
  // kernels of decode_dp4a.cu stop there), so smaller matrices keep the
  // quantization + small-CTA codes kernel
  return K <= 8192 || packed_layout_bytes(N, K) >= kCcMinBytes;
}

size_t decode_cc_smem(int64_t M, int64_t K) {
  const int S = cc_stages(M, K);
  return S ? (size_t)kCcWarps * S * kItemBytes + (size_t)cc_staging(M, K) : 0;
}

cudaError_t launch_layer_cc(const uint16_t* x, const uint16_t* gain, float rms_eps, const uint8_t* packed,
                               const float* w_scale, int64_t M, int64_t N, int64_t K, int out_dtype, void* y,
                               int8_t* x_q, float* act_scale, int32_t* acc_debug, bool pdl, cudaStream_t stream,
                               L2Prefetch pf) {
  if (!fused_route(M, N, K)) return cudaErrorInvalidValue;
  if (packed_layout_bytes(N, K) < kCcMinBytes && dp4a_layer_ok(M, N, K))
    return launch_linear_dp4a(x, gain, rms_eps, packed, w_scale, N, K, out_dtype, y, x_q, act_scale, acc_debug, pdl,
                              stream, pf);
  DecodeCcParams p = {};
  p.packed = packed;
  p.w_scale = w_scale;
  p.y = y;
  p.acc_debug = acc_debug;
  p.pf = pf.p;
  p.pf_bytes = pf.bytes;
  p.x = reinterpret_cast<const uint4*>(x);
  p.gain = reinterpret_cast<const uint4*>(gain);
  p.rms_eps = rms_eps;
  p.x_q_out = x_q;
  p.act_scale_out = act_scale;
  p.dev_err = current_device_error_word();
  if (!p.dev_err) return cudaErrorInvalidDevice;
  p.out_dtype = out_dtype;
  return launch_cc(p, M, N, K, true, pdl, stream);
}

cudaError_t launch_codes_cc(const int8_t* x_q, const float* act_scale, const uint8_t* packed,
                               const float* w_scale, int64_t M, int64_t N, int64_t K, int out_dtype,
                               void* y, int32_t* acc_debug, bool pdl, cudaStream_t stream, L2Prefetch pf) {
  if (!codes_route(M, N, K)) return cudaErrorInvalidValue;
  if (packed_layout_bytes(N, K) < kCcMinBytes && dp4a_codes_ok(M, N, K))
    return launch_decode_dp4a(x_q, act_scale, packed, w_scale, M, N, K, out_dtype, y, acc_debug, pdl, stream, pf);
  DecodeCcParams p = {};
  p.packed = packed;
  p.w_scale = w_scale;
  p.y = y;
  p.acc_debug = acc_debug;
  p.pf = pf.p;
  p.pf_bytes = pf.bytes;
  p.x_q = x_q;
  p.act_scale = act_scale;
  p.out_dtype = out_dtype;
  return launch_cc(p, M, N, K, false, pdl, stream);
}

}  // namespace bitlinear
