// bitlinear_pack_weights_static: the weight packer for callers that cannot
// allocate device memory.
//
// bitlinear_pack_weights needs ~2 KB of scratch (the exponent bins of the exact
// absmean and the resulting gamma) and asks the caller for it.  Some callers
// cannot provide it: a plugin that only ever receives the buffers its host
// framework sized in advance, or code on a latency-critical path where
// cudaMalloc / cudaFree may synchronize the whole device or fail under memory
// pressure.  This entry point runs the very same kernels with the scratch in a
// fixed file-scope device array instead, so the call allocates nothing.
//
// Costs of that choice:
//   - every GPU that loads this library holds the array (kPackWorkspaceBytes
//     bytes) until the process exits;
//   - all calls on one device share the array, which keeps whatever the last
//     call left in it.  Each call clears the bins it accumulates into before
//     use, but two calls whose work overlaps on the GPU (different streams with
//     no ordering between them) race on the array and may return a wrong gamma;
//   - the first call on each device looks the array's device address up with
//     cudaGetSymbolAddress while that device is current.  Make that first call
//     before any stream capture.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "../../include/bitlinear.h"
#include "internal.h"

namespace bitlinear {
namespace {

// The scratch of the allocation-free packer, one copy per device.
static __device__ __align__(256) unsigned char g_pack_scratch[kPackWorkspaceBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {nullptr};

// Device address of g_pack_scratch on the current device, looked up once per
// device (host code cannot use the symbol itself: it names a host-side shadow).
void* scratch_on_current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_pack_scratch) != cudaSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    g_scratch_ptr[dev] = p;
  }
  return g_scratch_ptr[dev];
}

bool aligned16_(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace bitlinear

extern "C" bitlinear_status bitlinear_pack_weights_static(const float* W, int64_t N, int64_t K,
                                                          float eps, uint8_t* packed,
                                                          float* w_scale, float* gamma_out,
                                                          void* stream) {
  using namespace bitlinear;
  if (!W || !packed || !w_scale) return BITLINEAR_ERR_NULL;
  // N*K < 2^32 keeps every 64-bit exponent bin of the fixed scratch from overflowing.
  if (N < 1 || K < 4 || K % 4 != 0 || N * K >= (int64_t(1) << 32) || !(eps >= 0.0f))
    return BITLINEAR_ERR_SHAPE;
  if (!aligned16_(W) || !aligned16_(packed) || !aligned16_(w_scale) ||
      (gamma_out && !aligned16_(gamma_out)))
    return BITLINEAR_ERR_ALIGN;
  int* err_word = current_device_error_word();
  if (!err_word) return BITLINEAR_ERR_DEVICE;
  void* scratch = scratch_on_current_device();
  if (!scratch) return BITLINEAR_ERR_CUDA;
  const cudaError_t e = launch_pack_weights(W, N, K, eps, packed, w_scale, gamma_out, scratch,
                                            err_word, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? BITLINEAR_OK : BITLINEAR_ERR_CUDA;
}
