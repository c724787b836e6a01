// Decode contraction for one or two tokens on the CUDA cores: y = dequant(x_q . W_q^T)
// with four-way int8 dot products (dp4a).
//
// Page "BitNet b1.58 in Production: 1-Bit LLMs and Energy Benchmarks", section
// "The Mathematical Mechanism", items 3-4 (integer product, rescale by the two
// scales); page "BitNet 1-bit LLM Inference Framework", section "How the LUT
// Kernel Works" (the 2-bit code, integer accumulation of the ternary products).
//
// Why a second decode kernel: with one or two tokens a launch moves a few MB,
// and in a chain of kernels (quantization -> contraction -> ...) its latency
// after the dependency is what counts.  Here a CTA owns 16 weight rows; its
// threads load their rows' packed codes into registers before waiting for the
// previous kernel (weights are not written by in-flight work), then stage the
// tokens' int8 codes in shared memory, run the dot products and reduce over
// eight lanes: no tensor-memory allocation, no MMA pipeline and no cluster-wide
// reduction after the wait.
//
// Threads: a row is read by 8 KS lanes (KS = 1, 2 or 4, more for longer rows):
// lane (ks, c) reads the 16-byte chunk c (64 inputs) of segments ks, ks + KS,
// ... of the tile-major packed layout; a warp holds 4 / KS rows, a CTA 16 / KS.  A 32-bit word of
// codes (16 inputs) is expanded by byte permutes into int8 words of inputs
// (0,2,4,6), (8..14 even), (1,3,5,7), (9..15 odd) (code 0 -> 0, 1 -> +1,
// 2 -> -1); the staged activations are permuted the same way, so a word is four
// dp4a per token.  The int32 sums are exact (|acc| <= 128 K < 2^31).
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "act_ops.cuh"
#include "device_util.cuh"
#include "internal.h"
#include "quant_math.cuh"

namespace bitlinear {
namespace {

constexpr int kDThreads = 128;               // 4 warps
constexpr int kChunkPitch = 80;              // a staged 64-byte chunk + 16 bytes: conflict-free reads
constexpr int kSegPitch = 8 * kChunkPitch;   // one token's 512 inputs in shared memory
constexpr uint32_t kCodeToI8 = 0x00FF0100u;  // bytes 0x00 (code 0), 0x01 (+1), 0xFF (-1)
constexpr int kFusedMaxSeg = 16;             // the one-token layer kernel: K <= 8192

struct DecodeDp4aParams {
  const uint8_t* packed;
  const int8_t* x_q;
  const float* act_scale;
  const float* w_scale;
  void* y;
  int32_t* acc_debug;
  const uint8_t* pf;         // L2 prefetch of the caller (or null)
  uint64_t pf_bytes;
  int M, N, K, nseg, Np, out_dtype;
};

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

// MT: tokens (1 or 2).  KS: lanes per (row, chunk) = 8 KS lanes per
// row, lane ks taking segments ks, ks + KS, ...  PRE: segments per lane loaded
// before the wait (later ones are read after it).
template <int MT, int KS, int PRE>
__global__ void __launch_bounds__(kDThreads) decode_dp4a_kernel(const DecodeDp4aParams p) {
  extern __shared__ __align__(16) uint8_t xsm[];
  constexpr int kRowsPerWarp = 4 / KS;
  constexpr int kLog2KS = KS == 1 ? 0 : KS == 2 ? 1 : 2;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = lane & 7;                                        // chunk of a segment
  const int ks = (lane >> 3) & (KS - 1);                         // first segment of this lane
  const int row = (blockIdx.x * 4 + warp) * kRowsPerWarp + (lane >> (3 + kLog2KS));   // < Np
  const int tile = row >> 7, r = row & 127;
  const int R = min(128, p.Np - tile * 128);                     // rows of this tile
  // chunk c of row r in segment s: tile base + s * R * 128 + r * 128, stored at c ^ (r % 8)
  const uint8_t* wrow = p.packed + (size_t)tile * p.nseg * 16384 + (size_t)r * 128 + ((c ^ (r & 7)) << 4);
  const size_t seg_step = (size_t)R * 128;

  uint4 wreg[PRE];
#pragma unroll
  for (int i = 0; i < PRE; ++i) {
    const int s = ks + KS * i;
    wreg[i] = s < p.nseg ? __ldg(reinterpret_cast<const uint4*>(wrow + s * seg_step)) : make_uint4(0u, 0u, 0u, 0u);
  }
  const bool nv = row < p.N;
  const float wsn = nv ? __ldg(p.w_scale + row) : 0.0f;
  if (threadIdx.x < 32) l2_prefetch_share(p.pf, p.pf_bytes, threadIdx.x, 32);
  pdl_launch_dependents();
  pdl_wait();                                // x_q, act_scale and y follow the stream order

  // this lane's output (token c of its row, written by the lanes with ks == 0)
  const bool out = nv && ks == 0 && c < p.M;
  const float as = out ? __ldcg(p.act_scale + c) : 0.0f;
  float res = 0.0f;
  if (out && p.out_dtype == 2)
    res = __uint_as_float((uint32_t)__ldcg(reinterpret_cast<const unsigned short*>(p.y) + (size_t)c * p.N + row) << 16);

  // stage the tokens' codes, permuted per 16 inputs; zeros past K and past M
  const int groups = p.nseg * 32;            // 16-input groups per token (Kp / 16)
  const uint32_t tstride = (uint32_t)(p.nseg * kSegPitch);
  for (int i = threadIdx.x; i < MT * groups; i += kDThreads) {
    const int m = i / groups, g = i - m * groups;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (m < p.M && 16 * g < p.K) v = __ldcg(reinterpret_cast<const uint4*>(p.x_q + (size_t)m * p.K) + g);
    const int s = g >> 5, cc = (g >> 2) & 7, j = g & 3;
    *reinterpret_cast<uint4*>(xsm + m * tstride + s * kSegPitch + cc * kChunkPitch + 16 * j) = permute16(v);
  }
  __syncthreads();

  int acc[MT];
#pragma unroll
  for (int m = 0; m < MT; ++m) acc[m] = 0;
  const uint32_t xs = smem_u32(xsm) + c * kChunkPitch;
#pragma unroll
  for (int i = 0; i < PRE; ++i) {
    const int s = ks + KS * i;
    if (s < p.nseg) dot_chunk<MT>(wreg[i], xs + s * kSegPitch, tstride, acc);
  }
  for (int s = ks + KS * PRE; s < p.nseg; s += KS)
    dot_chunk<MT>(__ldg(reinterpret_cast<const uint4*>(wrow + s * seg_step)), xs + s * kSegPitch, tstride, acc);

  // sum over the row's 8 KS lanes; lane (ks = 0, c) keeps token c
  int mine = 0;
#pragma unroll
  for (int m = 0; m < MT; ++m) {
    int v = acc[m];
#pragma unroll
    for (int o = 1; o < 8 * KS; o <<= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (m == c) mine = v;
  }
  if (!out) return;
  const size_t o = (size_t)c * p.N + row;
  const float yv = __fmul_rn(__fmul_rn((float)mine, as), wsn);
  if (p.out_dtype == 0) reinterpret_cast<float*>(p.y)[o] = yv;
  else if (p.out_dtype == 1) reinterpret_cast<__nv_bfloat16*>(p.y)[o] = __float2bfloat16_rn(yv);
  else reinterpret_cast<__nv_bfloat16*>(p.y)[o] = __float2bfloat16_rn(__fadd_rn(res, yv));
  if (p.acc_debug) p.acc_debug[o] = mine;
}

template <int MT, int KS, int PRE>
cudaError_t launch_cfg(const DecodeDp4aParams& p, size_t smem, bool pdl, cudaStream_t stream) {
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(decode_dp4a_kernel<MT, KS, PRE>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(p.Np * KS / 16), 1, 1);        // 16 / KS rows per CTA
  cfg.blockDim = dim3(kDThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, decode_dp4a_kernel<MT, KS, PRE>, p);
}

template <int MT, int KS>
cudaError_t launch_ks(const DecodeDp4aParams& p, size_t smem, bool pdl, cudaStream_t stream) {
  return (p.nseg + KS - 1) / KS <= 4 ? launch_cfg<MT, KS, 4>(p, smem, pdl, stream)
                                     : launch_cfg<MT, KS, 8>(p, smem, pdl, stream);
}

template <int MT>
cudaError_t launch_mt(const DecodeDp4aParams& p, int KS, size_t smem, bool pdl, cudaStream_t stream) {
  if (KS == 4) return launch_ks<MT, 4>(p, smem, pdl, stream);
  if (KS == 2) return launch_ks<MT, 2>(p, smem, pdl, stream);
  return launch_ks<MT, 1>(p, smem, pdl, stream);
}

// ---- the whole layer for one token: RMSNorm + quantization + contraction --------
// Every CTA forms the token's statistics itself (max|x g| and the pair sum of x^2)
// with the thread-to-input mapping and reduction tree of quant_act_kernel for one
// row (thread u takes inputs 16u..16u+15; its warps past the row add zeros, which
// leaves the tree's result unchanged), so codes and scale equal that kernel's bit
// for bit; the codes then go straight into the staging of the contraction.  CTA 0
// also writes x_q and act_scale when asked for.  T = blockDim.x >= Kp / 16.

struct LinearDp4aParams {
  const uint4* x;            // bf16 row, 8 per vector
  const uint4* gain;         // bf16 [K] or null
  float rms_eps;
  const uint8_t* packed;
  const float* w_scale;
  void* y;
  int8_t* x_q;               // [K] out, or null
  float* act_scale;          // [1] out, or null
  int32_t* acc_debug;
  const uint8_t* pf;         // L2 prefetch of the caller (or null)
  uint64_t pf_bytes;
  int N, K, nseg, Np, out_dtype;
};

template <int KS, int PRE>
__global__ void __launch_bounds__(512) linear_dp4a_kernel(const LinearDp4aParams p) {
  __shared__ __align__(16) uint8_t xsm[kFusedMaxSeg * kSegPitch];
  __shared__ float s_max[32];
  __shared__ float2 s_ss[32];
  __shared__ float s_m, s_sum;
  constexpr int kRowsPerWarp = 4 / KS;
  constexpr int kLog2KS = KS == 1 ? 0 : KS == 2 ? 1 : 2;
  const int tid = threadIdx.x, T = blockDim.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int c = lane & 7;
  const int ks = (lane >> 3) & (KS - 1);
  const int row = (blockIdx.x * (T >> 5) + warp) * kRowsPerWarp + (lane >> (3 + kLog2KS));
  const bool rv = row < p.Np;                                    // the last CTA may reach past Np
  const int tile = row >> 7, r = row & 127;
  const int R = min(128, p.Np - tile * 128);
  const uint8_t* wrow = p.packed + (size_t)tile * p.nseg * 16384 + (size_t)r * 128 + ((c ^ (r & 7)) << 4);
  const size_t seg_step = (size_t)R * 128;
  uint4 wreg[PRE];
#pragma unroll
  for (int i = 0; i < PRE; ++i) {
    const int s = ks + KS * i;
    wreg[i] = (rv && s < p.nseg) ? __ldg(reinterpret_cast<const uint4*>(wrow + s * seg_step))
                                 : make_uint4(0u, 0u, 0u, 0u);
  }
  const bool nv = row < p.N;
  const float wsn = nv ? __ldg(p.w_scale + row) : 0.0f;
  // this thread's unit of the token: inputs 16 tid .. 16 tid + 15 (vectors 2 tid, 2 tid + 1)
  const int V = p.K >> 3, U = (V + 1) >> 1;
  uint4 gv[2];
#pragma unroll
  for (int hv = 0; hv < 2; ++hv) {
    const int v = 2 * tid + hv;
    gv[hv] = (p.gain && tid < U && v < V) ? __ldg(p.gain + v) : kOnes;
  }
  if (tid < U && (tid & 3) == 0) prefetch_l2(p.x + 2 * tid);
  if (tid < 32) l2_prefetch_share(p.pf, p.pf_bytes, tid, 32);
  pdl_launch_dependents();
  pdl_wait();                                // x and y follow the stream order

  const bool out = nv && ks == 0 && c == 0;
  float res = 0.0f;
  if (out && p.out_dtype == 2)
    res = __uint_as_float((uint32_t)__ldcg(reinterpret_cast<const unsigned short*>(p.y) + row) << 16);

  // statistics, as quant_act_kernel
  uint4 xv[2];
  float amax = 0.0f, hi = 0.0f, lo = 0.0f;
#pragma unroll
  for (int hv = 0; hv < 2; ++hv) {
    const int v = 2 * tid + hv;
    if (tid < U && v < V) {
      xv[hv] = __ldcg(p.x + v);
      float xf[8], gf[8];
      unpack8(xv[hv], xf);
      unpack8(gv[hv], gf);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        amax = fmaxf(amax, fabsf(__fmul_rn(xf[j], gf[j])));
        float s_, e_;
        two_sum(hi, __fmul_rn(xf[j], xf[j]), s_, e_);
        hi = s_;
        lo = __fadd_rn(lo, e_);
      }
    } else {
      xv[hv] = make_uint4(0u, 0u, 0u, 0u);
    }
  }
  block_stats(amax, hi, lo, tid, T >> 5, s_max, s_ss, &s_m, &s_sum);
  const RowQuant rq = row_quant(s_m, s_sum, p.K, p.rms_eps);
  const float sigma = rq.sigma;

  // codes of this unit (zero past K), staged permuted for the dot products
  if (tid < p.nseg * 32) {
    uint32_t w[4];
    row_codes<16>([&](int j) { return __fmul_rn(bf16_at(xv[j >> 3], j & 7), bf16_at(gv[j >> 3], j & 7)); }, rq, w);
    const uint4 codes = make_uint4(w[0], w[1], w[2], w[3]);
    const int s = tid >> 5, cc = (tid >> 2) & 7, j = tid & 3;
    *reinterpret_cast<uint4*>(xsm + s * kSegPitch + cc * kChunkPitch + 16 * j) = permute16(codes);
    if (blockIdx.x == 0 && p.x_q && tid < U) *reinterpret_cast<uint4*>(p.x_q + 16 * tid) = codes;
  }
  if (blockIdx.x == 0 && tid == 0 && p.act_scale) *p.act_scale = sigma;
  __syncthreads();

  int acc[1] = {0};
  const uint32_t xs = smem_u32(xsm) + c * kChunkPitch;
#pragma unroll
  for (int i = 0; i < PRE; ++i) {
    const int s = ks + KS * i;
    if (s < p.nseg) dot_chunk<1>(wreg[i], xs + s * kSegPitch, 0u, acc);
  }
  for (int s = ks + KS * PRE; s < p.nseg; s += KS)
    dot_chunk<1>(rv ? __ldg(reinterpret_cast<const uint4*>(wrow + s * seg_step)) : make_uint4(0u, 0u, 0u, 0u),
                 xs + s * kSegPitch, 0u, acc);
  int v = acc[0];
#pragma unroll
  for (int o = 1; o < 8 * KS; o <<= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  if (!out) return;
  const float yv = __fmul_rn(__fmul_rn((float)v, sigma), wsn);
  if (p.out_dtype == 0) reinterpret_cast<float*>(p.y)[row] = yv;
  else if (p.out_dtype == 1) reinterpret_cast<__nv_bfloat16*>(p.y)[row] = __float2bfloat16_rn(yv);
  else reinterpret_cast<__nv_bfloat16*>(p.y)[row] = __float2bfloat16_rn(__fadd_rn(res, yv));
  if (p.acc_debug) p.acc_debug[row] = v;
}

template <int KS, int PRE>
cudaError_t launch_fused_cfg(const LinearDp4aParams& p, int T, bool pdl, cudaStream_t stream) {
  const int rows = (T / 32) * 4 / KS;                            // weight rows per CTA
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((p.Np + rows - 1) / rows), 1, 1);
  cfg.blockDim = dim3((unsigned)T, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, linear_dp4a_kernel<KS, PRE>, p);
}

template <int KS>
cudaError_t launch_fused_ks(const LinearDp4aParams& p, int T, bool pdl, cudaStream_t stream) {
  const int per_lane = (p.nseg + KS - 1) / KS;
  return per_lane <= 4 ? launch_fused_cfg<KS, 4>(p, T, pdl, stream)
       : per_lane <= 6 ? launch_fused_cfg<KS, 6>(p, T, pdl, stream)
                       : launch_fused_cfg<KS, 8>(p, T, pdl, stream);
}

size_t decode_dp4a_smem(int64_t M, int64_t K) {
  return (size_t)((M <= 1 ? 1 : 2) * (act_ops_kpad(K) / 512) * kSegPitch);
}

// Lanes per (row, chunk): the fewest that leave a lane at most five segments (more
// lanes and CTAs cost time where the rows are short: measured).
int dp4a_split(int nseg) {
  int ks = 1;
  while (ks < 4 && (nseg + ks - 1) / ks > 5) ks *= 2;
  return ks;
}

}  // namespace

// Shapes this file's kernels take: the codes kernel one token (any K) or two with
// K <= 4096 and N K <= 2^26, within its shared memory; the layer kernel one token
// with K <= 8192.
bool dp4a_codes_ok(int64_t M, int64_t N, int64_t K) {
  return (M == 1 || (M == 2 && K <= 4096 && N * K <= (int64_t(1) << 26))) &&
         decode_dp4a_smem(M, K) <= 227 * 1024;
}

bool dp4a_layer_ok(int64_t M, int64_t N, int64_t K) {
  return M == 1 && K <= kFusedMaxSeg * 512 && dp4a_codes_ok(M, N, K);
}

cudaError_t launch_linear_dp4a(const uint16_t* x, const uint16_t* gain, float rms_eps, const uint8_t* packed,
                               const float* w_scale, int64_t N, int64_t K, int out_dtype, void* y, int8_t* x_q,
                               float* act_scale, int32_t* acc_debug, bool pdl, cudaStream_t stream,
                               L2Prefetch pf) {
  if (!dp4a_layer_ok(1, N, K)) return cudaErrorInvalidValue;
  LinearDp4aParams p = {};
  p.x = reinterpret_cast<const uint4*>(x);
  p.gain = reinterpret_cast<const uint4*>(gain);
  p.rms_eps = rms_eps;
  p.packed = packed;
  p.w_scale = w_scale;
  p.y = y;
  p.x_q = x_q;
  p.act_scale = act_scale;
  p.acc_debug = acc_debug;
  p.pf = pf.p;
  p.pf_bytes = pf.bytes;
  p.N = (int)N;
  p.K = (int)K;
  p.nseg = (int)(act_ops_kpad(K) / 512);
  p.Np = (int)packed_rows(N);
  p.out_dtype = out_dtype;
  // threads: quant_act_kernel's for this row (one per 16 inputs, in whole warps),
  // rounded up to whole 4-warp groups of rows
  const int tq = (int)((K / 16 + 31) / 32 * 32);
  const int T = (tq + 127) / 128 * 128;
  const int KS = dp4a_split(p.nseg);
  cudaError_t e;
  if (KS == 4) e = launch_fused_ks<4>(p, T, pdl, stream);
  else if (KS == 2) e = launch_fused_ks<2>(p, T, pdl, stream);
  else e = launch_fused_ks<1>(p, T, pdl, stream);
  count_launches(1);
  return e;
}

cudaError_t launch_decode_dp4a(const int8_t* x_q, const float* act_scale, const uint8_t* packed,
                               const float* w_scale, int64_t M, int64_t N, int64_t K, int out_dtype,
                               void* y, int32_t* acc_debug, bool pdl, cudaStream_t stream, L2Prefetch pf) {
  if (!dp4a_codes_ok(M, N, K)) return cudaErrorInvalidValue;
  const size_t smem = decode_dp4a_smem(M, K);
  DecodeDp4aParams p = {};
  p.packed = packed;
  p.x_q = x_q;
  p.act_scale = act_scale;
  p.w_scale = w_scale;
  p.y = y;
  p.acc_debug = acc_debug;
  p.pf = pf.p;
  p.pf_bytes = pf.bytes;
  p.M = (int)M;
  p.N = (int)N;
  p.K = (int)K;
  p.nseg = (int)(act_ops_kpad(K) / 512);
  p.Np = (int)packed_rows(N);
  p.out_dtype = out_dtype;
  const int KS = dp4a_split(p.nseg);
  const cudaError_t e = M <= 1 ? launch_mt<1>(p, KS, smem, pdl, stream) : launch_mt<2>(p, KS, smem, pdl, stream);
  count_launches(1);
  return e;
}

}  // namespace bitlinear
