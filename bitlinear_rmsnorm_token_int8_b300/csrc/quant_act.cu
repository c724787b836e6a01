// Fused RMSNorm + per-token absmax int8 activation quantization.
//
// Page "BitNet b1.58 in Production: 1-Bit LLMs and Energy Benchmarks":
//   section "The Mathematical Mechanism", item 2 (absmax, Q_b = 127, per token),
//   item 4 (the activation scale max|x|/Q_b enters the dequantization), and
//   bit_linear.py BitLinear.forward (nn.RMSNorm before activation_quant).
//
// One CTA per token row.  The row is read once from HBM with 16-byte loads and
// kept in registers; a block reduction gives max|x*g| (exact: max is order
// free) and sum x^2.  No fp64 is used (it is slow on this GPU): x^2 is exact in
// fp32 (bf16 squared), and the sum is carried as an unevaluated pair hi + lo
// of fp32 numbers with error-free additions (Knuth's TwoSum), i.e. to about
// 2^-44 relative, before it is rounded once to fp32.
//
// sigma = max|x*g| * r / 127 with r = 1/sqrt(sum/K + eps): every step is one
// IEEE round-to-nearest operation, so with u = 2^-24 the result is within
// 3.5 u (2.1e-7) of the exact value: sum u, /K 2u, +eps 3u, sqrt 2u, 1/ 2.5u,
// *m 3u, /127 3.5u.
//
// Clamp (activation_quant clamps max|x_norm| at 1e-8): a row whose max|n|,
// formed as fl(max|x*g| * r), is below 1e-8 takes 1e-8 as its max; its codes
// are rint(fl(fl(p * r) * fl(127 / 1e-8))) and sigma = fl(1e-8 / 127)
// (quant_math.cuh, row_quant).  Only rows of zeros or of tiny values reach it.
//
// Codes of the other rows.  r > 0 is one number per row, so Round(127 n/max|n|) with n = x*r*g
// equals Round(127 p/max|p|) with p = x*g, and p is exact in fp32 (two 8-bit
// significands).  The kernel forms t = p * fl(127/m) (relative error <= 2^-23,
// i.e. |t - 127p/m| < 1.6e-5) and takes rint(t) unless t lies within 2^-15 of
// a half-integer.  There it decides on the sign of 127 p - (floor(t) + 1/2) m:
// 127 p is exact (at most 16 + 7 significant bits), and one fused multiply-add
// forms the difference with a single rounding, which cannot change its sign;
// an exact zero is a tie and goes to the even code.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "act_ops.cuh"
#include "device_util.cuh"
#include "internal.h"
#include "quant_math.cuh"

namespace bitlinear {
namespace {

// Eight inputs of the gated MLP branch: h = bf16(fl(fl(max(gate, 0)^2) * up)),
// from fp32 rows [gate (K) | up (K)], packed as bf16 pairs like an input vector.
__device__ __forceinline__ uint4 relu2_gate8(const float* __restrict__ gu_row, int K, int v) {
  const float4* g4 = reinterpret_cast<const float4*>(gu_row + 8 * v);
  const float4* u4 = reinterpret_cast<const float4*>(gu_row + K + 8 * v);
  const float4 ga = __ldcg(g4), gb = __ldcg(g4 + 1), ua = __ldcg(u4), ub = __ldcg(u4 + 1);
  const float g[8] = {ga.x, ga.y, ga.z, ga.w, gb.x, gb.y, gb.z, gb.w};
  const float u[8] = {ua.x, ua.y, ua.z, ua.w, ub.x, ub.y, ub.z, ub.w};
  uint32_t w[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    uint32_t pair = 0;
#pragma unroll
    for (int b = 0; b < 2; ++b) {
      const float r = fmaxf(g[2 * j + b], 0.0f);
      const float h = __fmul_rn(__fmul_rn(r, r), u[2 * j + b]);
      pair |= (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(h)) << (16 * b);
    }
    w[j] = pair;
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// A thread owns units of 16 consecutive inputs (two 16-byte bf16 vectors), so
// that it can store the operand form of a unit with two 16-byte stores.
// Input: bf16 rows at x with a pitch of `ld` 16-byte vectors, or, when `glu` is
// set, the ReLU^2-gated product of fp32 [gate | up] rows of pitch 2K (see
// relu2_gate8).  x_q may be null (codes only in operand form).
template <int UPT>
__global__ void __launch_bounds__(1024)
quant_act_kernel(const uint4* __restrict__ x, int64_t ld, const float* __restrict__ glu,
                 const uint4* __restrict__ gain, float rms_eps,
                 int K, int8_t* __restrict__ x_q, float* __restrict__ act_scale,
                 uint8_t* __restrict__ x_ops, int64_t M) {
  const int V = K >> 3;                      // 16-byte vectors per row
  const int U = (V + 1) >> 1;                // units of 16 inputs
  const int row = blockIdx.x;
  const int tid = threadIdx.x;
  const int T = blockDim.x;
  // the RMSNorm gain is not written by earlier kernels: with few units per thread
  // (the short-M launch) load it before waiting; longer rows reload it in place
  constexpr bool kPreGain = UPT <= 2;
  uint4 gv_[kPreGain ? UPT : 1][2];
  if constexpr (kPreGain) {
#pragma unroll
    for (int i = 0; i < UPT; ++i)
#pragma unroll
      for (int hv = 0; hv < 2; ++hv) {
        const int v = 2 * (tid + i * T) + hv;
        gv_[i][hv] = (gain && tid + i * T < U && v < V) ? __ldg(gain + v) : kOnes;
      }
  }
  // Pull the row into L2 before the wait.  A row that no earlier kernel writes
  // (staged by a copy) then comes from L2 after the wait instead of HBM; a row that
  // the previous kernel writes is updated in L2, the point of coherence, so the
  // loads after the wait read its final values either way.
  const uint4* xr = x + (size_t)row * ld;
  if (!glu) {
#pragma unroll
    for (int i = 0; i < UPT; ++i) {
      const int u = tid + i * T;
      if (u < U && (u & 3) == 0) prefetch_l2(xr + 2 * u);   // one per 128-byte line
    }
  }
  // Let the next kernel launch now: it waits for this one to complete, and this one
  // completes only after the kernel before it (the wait below), so the next kernel
  // can set up and prefetch its weights while the previous one still runs.
  pdl_launch_dependents();
  pdl_wait();                                // x may be the previous kernel's output
  const float* gr = glu ? glu + (size_t)row * 2 * K : nullptr;

  uint4 xv[UPT][2];
  float amax = 0.0f;
  float hi = 0.0f, lo = 0.0f;                // sum of x^2 as hi + lo
#pragma unroll
  for (int i = 0; i < UPT; ++i) {
    const int u = tid + i * T;
#pragma unroll
    for (int hv = 0; hv < 2; ++hv) {
      const int v = 2 * u + hv;
      if (u < U && v < V) {
        xv[i][hv] = gr ? relu2_gate8(gr, K, v) : __ldcg(xr + v);
        float xf[8], gf[8];
        unpack8(xv[i][hv], xf);
        if constexpr (kPreGain) unpack8(gv_[i][hv], gf);
        else unpack8(gain ? __ldg(gain + v) : kOnes, gf);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          amax = fmaxf(amax, fabsf(__fmul_rn(xf[j], gf[j])));
          float s_, e_;
          two_sum(hi, __fmul_rn(xf[j], xf[j]), s_, e_);   // x^2 is exact in fp32
          hi = s_;
          lo = __fadd_rn(lo, e_);
        }
      } else {
        xv[i][hv] = make_uint4(0u, 0u, 0u, 0u);
      }
    }
  }

  // block reduction: max (exact) and the pair sum of squares
  __shared__ float s_max[32];
  __shared__ float2 s_ss[32];
  __shared__ float s_m;
  __shared__ float s_sum;
  block_stats(amax, hi, lo, tid, T >> 5, s_max, s_ss, &s_m, &s_sum);

  const RowQuant rq = row_quant(s_m, s_sum, K, rms_eps);
  if (tid == 0) act_scale[row] = rq.sigma;

  uint2* qr = reinterpret_cast<uint2*>(x_q + (size_t)row * K);
  const int64_t Kp = act_ops_kpad(K);
#pragma unroll
  for (int i = 0; i < UPT; ++i) {
    const int u = tid + i * T;
    if (u < U) {
      uint4 gu[2];
#pragma unroll
      for (int hv = 0; hv < 2; ++hv) {
        const int v = 2 * u + hv;
        if constexpr (kPreGain) gu[hv] = gv_[i][hv];
        else gu[hv] = (gain && v < V) ? __ldg(gain + v) : kOnes;
      }
      uint32_t w[4];
      row_codes<16>([&](int j) { return __fmul_rn(bf16_at(xv[i][j >> 3], j & 7), bf16_at(gu[j >> 3], j & 7)); },
                    rq, w);
#pragma unroll
      for (int hv = 0; hv < 2; ++hv)
        if (2 * u + hv < V && x_q) qr[2 * u + hv] = make_uint2(w[2 * hv], w[2 * hv + 1]);
      if (x_ops) write_act_ops16_any(x_ops, M, row, (int64_t)u << 4, Kp, w);   // zero x -> zero code
    }
  }
  if (x_ops) {                               // zero operands of the padding up to Kp
    const uint32_t z[4] = {0u, 0u, 0u, 0u};
    for (int u = U + tid; u < (int)(Kp >> 4); u += T) write_act_ops16_any(x_ops, M, row, (int64_t)u << 4, Kp, z);
  }
}

// Many rows (prefill): persistent CTAs, kRowsThreads threads each, take rows
// blockIdx.x, blockIdx.x + gridDim.x, ...  A row is staged in shared memory by
// one bulk copy into a double buffer, so the copy of the next row overlaps the
// work on this one; the gain is staged once.  Same arithmetic as
// quant_act_kernel, in two passes over the staged row.
constexpr int kRowsThreads = 256;
constexpr uint32_t kRowsSpin = 1u << 24;

__global__ void __launch_bounds__(kRowsThreads, 2)
quant_rows_kernel(const uint16_t* __restrict__ x, int64_t ld, const uint16_t* __restrict__ gain, float rms_eps,
                  int K, int8_t* __restrict__ x_q, float* __restrict__ act_scale, uint8_t* __restrict__ x_ops,
                  int64_t M, int* dev_err) {
  extern __shared__ __align__(16) uint8_t qsm[];
  const int rb = K * 2;                            // bytes of a row (a multiple of 16)
  const uint32_t buf0 = smem_u32(qsm), gbuf = buf0 + 2 * rb;
  __shared__ uint64_t bars[2];
  __shared__ float s_max[kRowsThreads / 32];
  __shared__ float2 s_ss[kRowsThreads / 32];
  __shared__ float s_m, s_sum;
  __shared__ int s_abort;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int V = K >> 3, U = (V + 1) >> 1;
  const int64_t Kp = act_ops_kpad(K);
  if (tid == 0) {
    mbar_init(smem_u32(&bars[0]), 1);
    mbar_init(smem_u32(&bars[1]), 1);
    s_abort = 0;
    fence_mbar_init();
  }
  // the gain is not written by earlier kernels: stage it before waiting for them
  for (int v = tid; v < V; v += kRowsThreads)
    *reinterpret_cast<uint4*>(qsm + 2 * rb + 16 * v) =
        gain ? __ldg(reinterpret_cast<const uint4*>(gain) + v) : kOnes;
  __syncthreads();
  pdl_launch_dependents();                         // as in quant_act_kernel
  pdl_wait();                                      // x may be the previous kernel's output
  // thread 0 issues the copies; `pend` = iteration whose copy is issued and not yet waited for
  int pend = -1;
  auto issue = [&](int64_t row, int iter) {
    const int b = iter & 1;
    mbar_arrive_expect_tx(smem_u32(&bars[b]), (uint32_t)rb);
    bulk_g2s(buf0 + b * rb, x + row * ld, (uint32_t)rb, smem_u32(&bars[b]));
  };
  if (tid == 0 && (int64_t)blockIdx.x < M) {
    issue(blockIdx.x, 0);
    pend = 0;
  }
  int it = 0;
  for (int64_t row = blockIdx.x; row < M; row += gridDim.x, ++it) {
    const int b = it & 1;
    if (tid == 0) {
      if (!mbar_wait_bounded(smem_u32(&bars[b]), (uint32_t)((it >> 1) & 1), kRowsSpin)) {
        atomicCAS(dev_err, 0, kDevErrTimeout);
        s_abort = 1;
      } else {
        pend = -1;
        if (row + gridDim.x < M) {                // the other buffer was released at the end of the last row
          issue(row + gridDim.x, it + 1);
          pend = it + 1;
        }
      }
    }
    __syncthreads();
    if (s_abort) break;
    if (!mbar_wait_bounded(smem_u32(&bars[b]), (uint32_t)((it >> 1) & 1), kRowsSpin)) break;  // complete: acquires the data
    const uint32_t xb = buf0 + b * rb;
    // pass 1: max |x g| (exact) and sum x^2 as an error-free pair
    float amax = 0.0f, hi = 0.0f, lo = 0.0f;
    for (int u = tid; u < U; u += kRowsThreads) {
#pragma unroll
      for (int hv = 0; hv < 2; ++hv) {
        const int v = 2 * u + hv;
        if (v < V) {
          float xf[8], gf[8];
          unpack8(lds128(xb + 16 * v), xf);
          unpack8(lds128(gbuf + 16 * v), gf);
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            amax = fmaxf(amax, fabsf(__fmul_rn(xf[j], gf[j])));
            float s_, e_;
            two_sum(hi, __fmul_rn(xf[j], xf[j]), s_, e_);
            hi = s_;
            lo = __fadd_rn(lo, e_);
          }
        }
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
      const float h2 = __shfl_xor_sync(0xffffffffu, hi, o), l2 = __shfl_xor_sync(0xffffffffu, lo, o);
      pair_add(hi, lo, h2, l2);
    }
    if (lane == 0) {
      s_max[warp] = amax;
      s_ss[warp] = make_float2(hi, lo);
    }
    __syncthreads();
    if (warp == 0) {
      float a = lane < kRowsThreads / 32 ? s_max[lane] : 0.0f;
      float2 p2 = lane < kRowsThreads / 32 ? s_ss[lane] : make_float2(0.0f, 0.0f);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
        const float h2 = __shfl_xor_sync(0xffffffffu, p2.x, o), l2 = __shfl_xor_sync(0xffffffffu, p2.y, o);
        pair_add(p2.x, p2.y, h2, l2);
      }
      if (lane == 0) {
        s_m = a;
        s_sum = __fadd_rn(p2.x, p2.y);
      }
    }
    __syncthreads();
    const RowQuant rq = row_quant(s_m, s_sum, K, rms_eps);
    if (tid == 0) act_scale[row] = rq.sigma;
    // pass 2: codes, the int8 row and the operand form
    uint2* qr = x_q ? reinterpret_cast<uint2*>(x_q + row * K) : nullptr;
    for (int u = tid; u < (int)(Kp >> 4); u += kRowsThreads) {
      uint32_t w[4];
#pragma unroll
      for (int hv = 0; hv < 2; ++hv) {
        const int v = 2 * u + hv;
        if (v < V) {
          const uint4 xw = lds128(xb + 16 * v), gw = lds128(gbuf + 16 * v);
          uint32_t w2[2];
          row_codes<8>([&](int j) { return __fmul_rn(bf16_at(xw, j), bf16_at(gw, j)); }, rq, w2);
          w[2 * hv] = w2[0];
          w[2 * hv + 1] = w2[1];
          if (qr) qr[v] = make_uint2(w2[0], w2[1]);
        } else {
          w[2 * hv] = w[2 * hv + 1] = 0u;            // padding up to Kp: zero operands
        }
      }
      if (x_ops) write_act_ops16_any(x_ops, M, row, (int64_t)u << 4, Kp, w);
    }
    __syncthreads();                               // buffer b is free for the row after next
  }
  // no copy may still be landing in shared memory when the CTA exits
  if (tid == 0 && pend >= 0 && !mbar_wait_bounded(smem_u32(&bars[pend & 1]), (uint32_t)((pend >> 1) & 1), kRowsSpin))
    atomicCAS(dev_err, 0, kDevErrTimeout);
}

}  // namespace

cudaError_t launch_quant_act(const uint16_t* x, const uint16_t* gain, float rms_eps, int64_t M,
                             int64_t K, int8_t* x_q, float* act_scale, uint8_t* x_ops, bool pdl,
                             cudaStream_t stream) {
  return launch_quant_act_ex(x, K, nullptr, gain, rms_eps, M, K, x_q, act_scale, x_ops, pdl, stream);
}

cudaError_t launch_quant_act_ex(const uint16_t* x, int64_t ld, const float* glu, const uint16_t* gain,
                                float rms_eps, int64_t M, int64_t K, int8_t* x_q, float* act_scale,
                                uint8_t* x_ops, bool pdl, cudaStream_t stream) {
  if (M == 0) return cudaSuccess;
  const int sms = num_sms();
  // Many long rows of bf16 input: persistent CTAs that stream rows through shared
  // memory.  Measured: faster from K > 4096 with at least four rows per SM; shorter
  // rows or fewer of them stay with one CTA per row.
  const int64_t rows_smem = 6 * K;            // two row buffers + the gain
  if (!glu && M >= 4 * sms && K > 4096 && rows_smem <= 100 * 1024) {
    int* dev_err = current_device_error_word();
    if (!dev_err) return cudaErrorInvalidDevice;
    static bool attr_set = false;
    if (!attr_set) {
      cudaError_t e = cudaFuncSetAttribute(quant_rows_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           100 * 1024);
      if (e != cudaSuccess) return e;
      attr_set = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(M < 2 * sms ? M : 2 * sms), 1, 1);
    cfg.blockDim = dim3(kRowsThreads, 1, 1);
    cfg.dynamicSmemBytes = (size_t)rows_smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    cudaError_t e = cudaLaunchKernelEx(&cfg, quant_rows_kernel, x, ld, gain, rms_eps, (int)K, x_q, act_scale,
                                       x_ops, M, dev_err);
    count_launches(1);
    return e;
  }
  const int U = (int)((K / 8 + 1) / 2);       // units of 16 inputs
  int T, vpt;
  // Few rows (decode): each row is one CTA's serial chain, so spread it over up
  // to 1024 threads.  Many rows: 256-thread CTAs keep many rows in flight.
  if (U <= 256) {
    T = ((U + 31) / 32) * 32;
    vpt = 1;
  } else if (M < sms || U > 1024) {
    T = U <= 1024 ? ((U + 31) / 32) * 32 : 1024;
    vpt = (U + T - 1) / T;
  } else {
    T = 256;
    vpt = (U + 255) / 256;
  }
  int tv = 1;
  while (tv < vpt) tv <<= 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)M, 1, 1);
  cfg.blockDim = dim3((unsigned)T, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  const uint4* xv = reinterpret_cast<const uint4*>(x);
  const uint4* gv = reinterpret_cast<const uint4*>(gain);
  cudaError_t e;
  switch (tv) {
    case 1: e = cudaLaunchKernelEx(&cfg, quant_act_kernel<1>, xv, (int64_t)(ld / 8), glu, gv, rms_eps, (int)K, x_q, act_scale, x_ops, M); break;
    case 2: e = cudaLaunchKernelEx(&cfg, quant_act_kernel<2>, xv, (int64_t)(ld / 8), glu, gv, rms_eps, (int)K, x_q, act_scale, x_ops, M); break;
    case 4: e = cudaLaunchKernelEx(&cfg, quant_act_kernel<4>, xv, (int64_t)(ld / 8), glu, gv, rms_eps, (int)K, x_q, act_scale, x_ops, M); break;
    default: e = cudaLaunchKernelEx(&cfg, quant_act_kernel<8>, xv, (int64_t)(ld / 8), glu, gv, rms_eps, (int)K, x_q, act_scale, x_ops, M); break;
  }
  count_launches(1);
  return e;
}

}  // namespace bitlinear
