// C ABI of libbitlinear: argument validation, per-device set-up, dispatch.
// The declarations and the contract of every entry point are in bitlinear.h.
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

#include "../../include/bitlinear.h"
#include "act_ops.cuh"
#include "internal.h"

namespace bitlinear {

// Per-device error word written by kernels (first error wins, atomicCAS from 0).
__device__ int g_device_error;

namespace {

constexpr int kMaxDevices = 64;

struct DeviceState {
  bool ready = false;
  bool ok = false;
  int sms = 0;
  int* err_word = nullptr;   // device address of g_device_error on this device
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];

// Checks the current device once (compute capability 10.3) and caches its SM
// count and the device address of the error word.
const DeviceState* current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState& s = g_dev[dev];
  if (!s.ready) {
    s.ready = true;
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    void* p = nullptr;
    if (major == 10 && minor == 3 && cudaGetSymbolAddress(&p, g_device_error) == cudaSuccess) {
      s.ok = true;
      s.sms = sms;
      s.err_word = static_cast<int*>(p);
    }
    cudaGetLastError();
  }
  return s.ok ? &s : nullptr;
}

constexpr unsigned kKnownFlags = BITLINEAR_FLAG_PDL;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bitlinear_status from_cuda(cudaError_t e) {
  return e == cudaSuccess ? BITLINEAR_OK : BITLINEAR_ERR_CUDA;
}

// The caller's L2 prefetch range, its size rounded down to 16 bytes (empty when
// either is 0 / NULL).
L2Prefetch prefetch_range(const void* p, size_t bytes) {
  L2Prefetch pf;
  if (p && bytes >= 16) {
    pf.p = static_cast<const uint8_t*>(p);
    pf.bytes = (uint64_t)(bytes & ~size_t(15));
  }
  return pf;
}

}  // namespace

static std::atomic<uint64_t> g_launches{0};

void count_launches(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }

int* current_device_error_word() {
  const DeviceState* s = current_device();
  return s ? s->err_word : nullptr;
}

int num_sms() {
  const DeviceState* s = current_device();
  return s ? s->sms : 148;
}

}  // namespace bitlinear

using namespace bitlinear;

extern "C" {

const char* bitlinear_status_string(bitlinear_status status) {
  switch (status) {
    case BITLINEAR_OK: return "ok";
    case BITLINEAR_ERR_NULL: return "null pointer";
    case BITLINEAR_ERR_SHAPE: return "invalid shape";
    case BITLINEAR_ERR_ALIGN: return "pointer not 16-byte aligned";
    case BITLINEAR_ERR_DTYPE: return "invalid output dtype";
    case BITLINEAR_ERR_DEVICE: return "current device is not an sm_103 GPU";
    case BITLINEAR_ERR_CUDA: return "CUDA error";
    case BITLINEAR_ERR_TIMEOUT: return "bounded wait timed out on the device";
    case BITLINEAR_ERR_WORKSPACE: return "workspace missing or too small";
    case BITLINEAR_ERR_NONFINITE: return "non-finite latent weight";
    case BITLINEAR_ERR_FLAGS: return "unknown flag bits";
  }
  return "unknown status";
}

int bitlinear_abi_version(void) { return 2; }

uint64_t bitlinear_kernel_launches(void) { return g_launches.load(std::memory_order_relaxed); }

size_t bitlinear_packed_bytes(int64_t N, int64_t K) {
  if (N < 1 || K < 4 || K % 4 != 0 || N > (int64_t(1) << 32) || K > (int64_t(1) << 32)) return 0;
  return (size_t)packed_layout_bytes(N, K);
}

size_t bitlinear_pack_workspace_bytes(int64_t, int64_t) { return kPackWorkspaceBytes; }

bitlinear_status bitlinear_pack_weights(const float* W, int64_t N, int64_t K, float eps,
                                        uint8_t* packed, float* w_scale, float* gamma_out,
                                        void* workspace, size_t workspace_bytes, void* stream) {
  if (!W || !packed || !w_scale) return BITLINEAR_ERR_NULL;
  if (N < 1 || K < 4 || K % 4 != 0 || N * K >= (int64_t(1) << 32) || !(eps >= 0.0f))
    return BITLINEAR_ERR_SHAPE;
  if (!workspace || workspace_bytes < kPackWorkspaceBytes) return BITLINEAR_ERR_WORKSPACE;
  if (!aligned16(W) || !aligned16(packed) || !aligned16(w_scale) || !aligned16(workspace) ||
      (gamma_out && !aligned16(gamma_out)))
    return BITLINEAR_ERR_ALIGN;
  const DeviceState* dev = current_device();
  if (!dev) return BITLINEAR_ERR_DEVICE;
  return from_cuda(launch_pack_weights(W, N, K, eps, packed, w_scale, gamma_out, workspace,
                                       dev->err_word, static_cast<cudaStream_t>(stream)));
}

size_t bitlinear_act_ops_bytes(int64_t M, int64_t K) {
  if (M < 0 || K < 1) return 0;
  return act_ops_bytes(M, K);
}

bitlinear_status bitlinear_quant_act(const void* x_bf16, const void* gain_bf16, float rms_eps,
                                     int64_t M, int64_t K, int8_t* x_q, float* act_scale,
                                     void* x_ops, unsigned flags, void* stream) {
  if (M < 0 || M > (int64_t(1) << 31) - 1 || K < 8 || K > 65536 || K % 8 != 0)
    return BITLINEAR_ERR_SHAPE;
  if (flags & ~kKnownFlags) return BITLINEAR_ERR_FLAGS;
  if (M == 0) return BITLINEAR_OK;
  if (!x_bf16 || !x_q || !act_scale) return BITLINEAR_ERR_NULL;
  if (!aligned16(x_bf16) || !aligned16(x_q) || !aligned16(act_scale) ||
      (gain_bf16 && !aligned16(gain_bf16)) || (x_ops && !aligned16(x_ops)))
    return BITLINEAR_ERR_ALIGN;
  const DeviceState* dev = current_device();
  if (!dev) return BITLINEAR_ERR_DEVICE;
  return from_cuda(launch_quant_act(static_cast<const uint16_t*>(x_bf16),
                                    static_cast<const uint16_t*>(gain_bf16), rms_eps, M, K, x_q,
                                    act_scale, static_cast<uint8_t*>(x_ops),
                                    (flags & BITLINEAR_FLAG_PDL) != 0,
                                    static_cast<cudaStream_t>(stream)));
}

bitlinear_status bitlinear_pack_weights_per_channel(const float* W, int64_t N, int64_t K, float eps,
                                                    uint8_t* packed, float* w_scale, void* stream) {
  if (!W || !packed || !w_scale) return BITLINEAR_ERR_NULL;
  if (N < 1 || K < 4 || K % 4 != 0 || N * K >= (int64_t(1) << 32) || !(eps >= 0.0f))
    return BITLINEAR_ERR_SHAPE;
  if (!aligned16(W) || !aligned16(packed) || !aligned16(w_scale)) return BITLINEAR_ERR_ALIGN;
  const DeviceState* dev = current_device();
  if (!dev) return BITLINEAR_ERR_DEVICE;
  return from_cuda(launch_pack_weights_per_channel(W, N, K, eps, packed, w_scale, dev->err_word,
                                                   static_cast<cudaStream_t>(stream)));
}

size_t bitlinear_quant_act_per_tensor_workspace_bytes(int64_t M) {
  if (M < 0) return 0;
  return (size_t)((4 * M + 255) / 256 * 256);
}

bitlinear_status bitlinear_quant_act_per_tensor(const void* x_bf16, int64_t M, int64_t K, int8_t* x_q,
                                                float* act_scale, void* x_ops, void* workspace,
                                                size_t workspace_bytes, unsigned flags, void* stream) {
  if (M < 0 || M > (int64_t(1) << 31) - 1 || K < 8 || K > 65536 || K % 8 != 0)
    return BITLINEAR_ERR_SHAPE;
  if (flags & ~kKnownFlags) return BITLINEAR_ERR_FLAGS;
  if (M == 0) return BITLINEAR_OK;
  if (!x_bf16 || !x_q || !act_scale) return BITLINEAR_ERR_NULL;
  if (!aligned16(x_bf16) || !aligned16(x_q) || !aligned16(act_scale) || (x_ops && !aligned16(x_ops)))
    return BITLINEAR_ERR_ALIGN;
  if (!workspace || workspace_bytes < bitlinear_quant_act_per_tensor_workspace_bytes(M))
    return BITLINEAR_ERR_WORKSPACE;
  if (!aligned16(workspace)) return BITLINEAR_ERR_ALIGN;
  const DeviceState* dev = current_device();
  if (!dev) return BITLINEAR_ERR_DEVICE;
  return from_cuda(launch_quant_act_per_tensor(static_cast<const uint16_t*>(x_bf16), M, K, x_q, act_scale,
                                               static_cast<uint8_t*>(x_ops), static_cast<float*>(workspace),
                                               (flags & BITLINEAR_FLAG_PDL) != 0,
                                               static_cast<cudaStream_t>(stream)));
}

size_t bitlinear_forward_workspace_bytes(int64_t M, int64_t N, int64_t K) {
  if (M < 0 || N < 1 || K < 1) return 0;
  return forward_workspace_bytes(M, N, K);
}

static_assert(kCodesMaxM == BITLINEAR_CODES_MAX_M, "the header's CODES_MAX_M is the codes kernel's limit");

bitlinear_status bitlinear_forward(const int8_t* x_q, const float* act_scale, const void* x_ops,
                                   const uint8_t* packed, const float* w_scale, int64_t M,
                                   int64_t N, int64_t K, int out_dtype, void* y,
                                   int32_t* acc_debug, void* workspace, size_t workspace_bytes,
                                   const void* l2_prefetch, size_t l2_prefetch_bytes, unsigned flags,
                                   void* stream) {
  if (M < 0 || M > (int64_t(1) << 24) || N < 16 || N % 16 != 0 || N > (int64_t(1) << 24) ||
      K < 128 || K % 128 != 0 || K > 65536)
    return BITLINEAR_ERR_SHAPE;
  if (out_dtype != BITLINEAR_OUT_F32 && out_dtype != BITLINEAR_OUT_BF16 && out_dtype != BITLINEAR_OUT_BF16_ADD)
    return BITLINEAR_ERR_DTYPE;
  if (flags & ~kKnownFlags) return BITLINEAR_ERR_FLAGS;
  if (M == 0) return BITLINEAR_OK;
  if (!act_scale || !packed || !w_scale || !y || (!x_q && !x_ops)) return BITLINEAR_ERR_NULL;
  if ((x_q && !aligned16(x_q)) || (x_ops && !aligned16(x_ops)) || !aligned16(act_scale) ||
      !aligned16(packed) || !aligned16(w_scale) || !aligned16(y) ||
      (acc_debug && !aligned16(acc_debug)) || (l2_prefetch && !aligned16(l2_prefetch)))
    return BITLINEAR_ERR_ALIGN;
  if (!x_ops) {                                   // x_q is converted in the workspace, if needed
    const size_t need = forward_workspace_bytes(M, N, K);
    if (need && (!workspace || workspace_bytes < need)) return BITLINEAR_ERR_WORKSPACE;
    if (!aligned16(workspace)) return BITLINEAR_ERR_ALIGN;
  }
  const DeviceState* dev = current_device();
  if (!dev) return BITLINEAR_ERR_DEVICE;
  return from_cuda(launch_forward(x_q, act_scale, static_cast<const uint8_t*>(x_ops), packed,
                                  w_scale, M, N, K, out_dtype, y, acc_debug, workspace,
                                  dev->err_word, (flags & BITLINEAR_FLAG_PDL) != 0,
                                  static_cast<cudaStream_t>(stream), prefetch_range(l2_prefetch, l2_prefetch_bytes)));
}

namespace {
// Workspace of bitlinear_linear_forward when it runs as quantization + contraction:
// [0, ops) the operand form of the codes, [ops, ops + 4 M) the per-token scales.
size_t linear_ops_bytes(int64_t M, int64_t K) { return (act_ops_bytes(M, K) + 255) / 256 * 256; }
size_t linear_split_bytes(int64_t M, int64_t K) { return linear_ops_bytes(M, K) + (size_t)(4 * M + 255) / 256 * 256; }
}  // namespace

size_t bitlinear_linear_workspace_bytes(int64_t M, int64_t N, int64_t K) {
  if (M < 0 || N < 16 || N % 16 != 0 || K < 128 || K % 128 != 0 || K > 65536) return 0;
  return linear_split_bytes(M, K);
}

int bitlinear_linear_route(int64_t M, int64_t N, int64_t K) {
  if (M < 1 || M > (int64_t(1) << 24) || N < 16 || N % 16 != 0 || N > (int64_t(1) << 24) || K < 128 ||
      K % 128 != 0 || K > 65536)
    return -1;
  if (fused_route(M, N, K)) return BITLINEAR_ROUTE_FUSED;
  if (codes_route(M, N, K)) return BITLINEAR_ROUTE_CODES;
  return act_ops_prefill(M) ? BITLINEAR_ROUTE_PREFILL : BITLINEAR_ROUTE_DECODE;
}

int bitlinear_prefill_cluster_size(const void* x_ops, int64_t M, int64_t N, int64_t K) {
  if (bitlinear_linear_route(M, N, K) != BITLINEAR_ROUTE_PREFILL || !x_ops) return -1;
  return prefill_cluster(x_ops, N);
}

bitlinear_status bitlinear_linear_forward(const void* x_bf16, const void* gain_bf16, float rms_eps,
                                          const uint8_t* packed, const float* w_scale, int64_t M,
                                          int64_t N, int64_t K, int out_dtype, void* y, int8_t* x_q,
                                          float* act_scale, int32_t* acc_debug, void* workspace,
                                          size_t workspace_bytes, const void* l2_prefetch,
                                          size_t l2_prefetch_bytes, unsigned flags, void* stream) {
  if (M < 0 || M > (int64_t(1) << 24) || N < 16 || N % 16 != 0 || N > (int64_t(1) << 24) ||
      K < 128 || K % 128 != 0 || K > 65536)
    return BITLINEAR_ERR_SHAPE;
  if (out_dtype != BITLINEAR_OUT_F32 && out_dtype != BITLINEAR_OUT_BF16 && out_dtype != BITLINEAR_OUT_BF16_ADD)
    return BITLINEAR_ERR_DTYPE;
  if (flags & ~kKnownFlags) return BITLINEAR_ERR_FLAGS;
  if (M == 0) return BITLINEAR_OK;
  if (!x_bf16 || !packed || !w_scale || !y) return BITLINEAR_ERR_NULL;
  if (!aligned16(x_bf16) || (gain_bf16 && !aligned16(gain_bf16)) || !aligned16(packed) ||
      !aligned16(w_scale) || !aligned16(y) || (x_q && !aligned16(x_q)) || (act_scale && !aligned16(act_scale)) ||
      (acc_debug && !aligned16(acc_debug)) || (l2_prefetch && !aligned16(l2_prefetch)))
    return BITLINEAR_ERR_ALIGN;
  if (!workspace || workspace_bytes < linear_split_bytes(M, K)) return BITLINEAR_ERR_WORKSPACE;
  if (!aligned16(workspace)) return BITLINEAR_ERR_ALIGN;
  const DeviceState* dev = current_device();
  if (!dev) return BITLINEAR_ERR_DEVICE;
  const bool pdl = (flags & BITLINEAR_FLAG_PDL) != 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* ops = static_cast<uint8_t*>(workspace);
  float* scale = act_scale ? act_scale : reinterpret_cast<float*>(ops + linear_ops_bytes(M, K));
  const L2Prefetch next = prefetch_range(l2_prefetch, l2_prefetch_bytes);
  if (fused_route(M, N, K))                      // one token: the whole layer in one kernel
    return from_cuda(launch_layer_cc(static_cast<const uint16_t*>(x_bf16), static_cast<const uint16_t*>(gain_bf16),
                                     rms_eps, packed, w_scale, M, N, K, out_dtype, y, x_q, act_scale, acc_debug,
                                     pdl, s, next));
  // Two kernels: quantization, then the contraction, which prefetches the caller's range.
  if (codes_route(M, N, K)) {
    // a few tokens: the contraction reads the int8 codes (kept in the workspace's
    // operand region unless x_q is given), not the operand form
    int8_t* codes = x_q ? x_q : reinterpret_cast<int8_t*>(ops);
    cudaError_t e = launch_quant_act(static_cast<const uint16_t*>(x_bf16), static_cast<const uint16_t*>(gain_bf16),
                                     rms_eps, M, K, codes, scale, nullptr, pdl, s);
    if (e != cudaSuccess) return from_cuda(e);
    return from_cuda(launch_forward(codes, scale, nullptr, packed, w_scale, M, N, K, out_dtype, y, acc_debug,
                                    nullptr, dev->err_word, true, s, next));
  }
  cudaError_t e = launch_quant_act(static_cast<const uint16_t*>(x_bf16), static_cast<const uint16_t*>(gain_bf16),
                                   rms_eps, M, K, x_q, scale, ops, pdl, s);
  if (e != cudaSuccess) return from_cuda(e);
  // the contraction follows a kernel of this library: overlapping with it is safe
  return from_cuda(launch_forward(nullptr, scale, ops, packed, w_scale, M, N, K, out_dtype, y, acc_debug,
                                  nullptr, dev->err_word, true, s, next));
}

bitlinear_status bitlinear_get_device_error(void* stream) {
  const DeviceState* dev = current_device();
  if (!dev) return BITLINEAR_ERR_DEVICE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int host = 0;
  if (cudaStreamSynchronize(s) != cudaSuccess) return BITLINEAR_ERR_CUDA;
  if (cudaMemcpyFromSymbol(&host, g_device_error, sizeof(int)) != cudaSuccess) return BITLINEAR_ERR_CUDA;
  if (host != 0) {
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_device_error, &zero, sizeof(int)) != cudaSuccess) return BITLINEAR_ERR_CUDA;
  }
  return static_cast<bitlinear_status>(host);
}

}  // extern "C"
