// Dense tensor-core peak rates on this GPU, measured by back-to-back MMAs whose
// operands stay on chip: the roofline denominators of the prefill contraction.
// Built into libbitlinear_probe.so (not part of the BitLinear C ABI); bench.py
// times the launches with CUDA events and converts MMAs to FLOP/s.
//
//   bitlinear_probe_tcgen05(kind, iters, ctas, &ms)
//     kind 0: tcgen05.mma kind::f8f6f4, e4m3 x e4m3 -> fp32, m128 n256 k32
//     kind 1: tcgen05.mma kind::f16,    bf16 x bf16 -> fp32, m128 n256 k16
//     One CTA per SM: A (128 x K) in tensor memory, B (256 x K) in shared memory
//     (128-byte swizzled rows, as the prefill kernel reads its operands), D in
//     tensor memory; one thread issues `iters` MMAs, then waits for them.
//   bitlinear_probe_mma_sync(kind, iters, ctas, &ms)
//     kind 0: mma.sync m16n8k32 s8 x s8 -> s32; kind 1: the same shape in e4m3 ->
//     f32.  8 warps per CTA, 8 independent accumulators per warp.
//
// Every wait is bounded; the result is the elapsed time of the launch.
#include <cuda_runtime.h>
#include <stdint.h>

#include "../device_util.cuh"

namespace bitlinear {
namespace {

constexpr uint32_t kProbeSpin = 1u << 26;

__device__ __forceinline__ void mma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                           uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

template <int KIND>
__global__ void __launch_bounds__(128, 1) tcgen05_peak_kernel(int iters, int* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  __shared__ uint64_t bar;
  __shared__ uint32_t s_tmem;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // B: 256 rows x 128 bytes of small exact values (e4m3 1.0 = 0x38, bf16 1.0 = 0x3f80)
  for (int i = threadIdx.x; i < 256 * 128 / 4; i += blockDim.x)
    reinterpret_cast<uint32_t*>(smem)[i] = KIND == 0 ? 0x38383838u : 0x3f803f80u;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(smem_u32(&s_tmem), 512);
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  // A: 32 columns at 256 (four k-steps of 8 columns), one lane quarter per warp
  uint32_t a[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) a[j] = KIND == 0 ? 0x38383838u : 0x3f803f80u;
  tmem_st32(tmem + ((uint32_t)(32 * warp) << 16) + 256, a);
  tmem_wait_st();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (threadIdx.x == 0) {
    const uint32_t idesc = KIND == 0 ? idesc_e4m3_f32(128, 256)
                                     : ((1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(256 >> 3) << 17) |
                                        ((uint32_t)(128 >> 4) << 24));
    const uint32_t b0 = smem_u32(smem);
    for (int i = 0; i < iters; ++i) {
      const int s = i & 3;                   // k-step within the 128-byte rows
      const uint64_t bd = smem_desc_sw128(b0 + 32 * s);
      if (KIND == 0) mma_f8f6f4_ts(tmem, tmem + 256 + 8 * s, bd, idesc, i > 0 ? 1u : 0u);
      else mma_f16_ts(tmem, tmem + 256 + 8 * s, bd, idesc, i > 0 ? 1u : 0u);
    }
    mma_commit(smem_u32(&bar));
    if (!mbar_wait_bounded(smem_u32(&bar), 0, kProbeSpin)) atomicExch(err, 1);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, 512);
  (void)lane;
}

template <int KIND>
__global__ void __launch_bounds__(256) mma_sync_peak_kernel(int iters, int* out) {
  int acc[8][4];
  float facc[8][4];
#pragma unroll
  for (int j = 0; j < 8; ++j)
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      acc[j][r] = 0;
      facc[j][r] = 0.0f;
    }
  const uint32_t a0 = 0x01010101u + threadIdx.x, b0 = 0x01010101u ^ threadIdx.x;
  for (int i = 0; i < iters; ++i) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (KIND == 0) {
        asm volatile(
            "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
            "{%0,%1,%2,%3};"
            : "+r"(acc[j][0]), "+r"(acc[j][1]), "+r"(acc[j][2]), "+r"(acc[j][3])
            : "r"(a0), "r"(a0 + j), "r"(a0), "r"(a0), "r"(b0), "r"(b0 + i));
      } else {
        asm volatile(
            "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
            "{%0,%1,%2,%3};"
            : "+f"(facc[j][0]), "+f"(facc[j][1]), "+f"(facc[j][2]), "+f"(facc[j][3])
            : "r"(0x38383838u), "r"(0x38383838u), "r"(0x38383838u), "r"(0x38383838u), "r"(0x38383838u),
              "r"(0x38383838u));
      }
    }
  }
  int s = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j)
#pragma unroll
    for (int r = 0; r < 4; ++r) s += acc[j][r] + (int)facc[j][r];
  if (s == 0x7fffffff) out[0] = s;           // keeps the work; practically never stores
}

template <typename Launch>
int time_launch(Launch launch, float* ms) {
  cudaEvent_t e0, e1;
  if (cudaEventCreate(&e0) != cudaSuccess || cudaEventCreate(&e1) != cudaSuccess) return (int)cudaGetLastError();
  launch();                                   // warm-up (module load, clocks)
  cudaEventRecord(e0);
  launch();
  cudaEventRecord(e1);
  cudaError_t e = cudaEventSynchronize(e1);
  if (e == cudaSuccess) e = cudaEventElapsedTime(ms, e0, e1);
  if (e == cudaSuccess) e = cudaGetLastError();
  cudaEventDestroy(e0);
  cudaEventDestroy(e1);
  return (int)e;
}

}  // namespace
}  // namespace bitlinear

using namespace bitlinear;

extern "C" int bitlinear_probe_tcgen05(int kind, int iters, int ctas, float* ms) {
  int* err = nullptr;
  if (cudaMalloc(&err, sizeof(int)) != cudaSuccess) return (int)cudaGetLastError();
  cudaMemset(err, 0, sizeof(int));
  const size_t smem = 120 * 1024;              // B takes 33 KB; the rest keeps one CTA per SM
  auto f = kind == 0 ? tcgen05_peak_kernel<0> : tcgen05_peak_kernel<1>;
  cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  int rc = time_launch([&] { f<<<ctas, 128, smem>>>(iters, err); }, ms);
  int host = 0;
  if (rc == 0 && cudaMemcpy(&host, err, sizeof(int), cudaMemcpyDeviceToHost) == cudaSuccess && host) rc = -1;
  cudaFree(err);
  return rc;
}

extern "C" int bitlinear_probe_mma_sync(int kind, int iters, int ctas, float* ms) {
  int* out = nullptr;
  if (cudaMalloc(&out, sizeof(int)) != cudaSuccess) return (int)cudaGetLastError();
  auto f = kind == 0 ? mma_sync_peak_kernel<0> : mma_sync_peak_kernel<1>;
  int rc = time_launch([&] { f<<<ctas, 256>>>(iters, out); }, ms);
  cudaFree(out);
  return rc;
}
