// Host-side declarations shared by the translation units of libbitlinear.
// Launchers validate nothing: api.cu checks every argument before calling them.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace bitlinear {

// Device status values written into the per-device error word (same numbers
// as the public bitlinear_status codes).
constexpr int kDevErrTimeout = 7;
constexpr int kDevErrNonFinite = 9;

// ---- pack_weights --------------------------------------------------------
// Workspace layout (bytes): [0, 2048) 256 uint64 exponent bins of sum|W|,
// [2048, 2056) gamma and d = fl32(gamma + eps) as two floats.
constexpr size_t kPackBinsBytes = 256 * sizeof(unsigned long long);
constexpr size_t kPackWorkspaceBytes = kPackBinsBytes + 16;

cudaError_t launch_pack_weights(const float* W, int64_t N, int64_t K, float eps, uint8_t* packed,
                                float* w_scale, float* gamma_out, void* workspace, int* dev_err,
                                cudaStream_t stream);

// ---- quant_act -----------------------------------------------------------
cudaError_t launch_quant_act(const uint16_t* x, const uint16_t* gain, float rms_eps, int64_t M,
                             int64_t K, int8_t* x_q, float* act_scale, cudaStream_t stream);

// ---- forward ---------------------------------------------------------------
size_t forward_workspace_bytes(int64_t M, int64_t N, int64_t K);

cudaError_t launch_forward(const int8_t* x_q, const float* act_scale, const uint8_t* packed,
                           const float* w_scale, int64_t M, int64_t N, int64_t K, int out_dtype,
                           void* y, int32_t* acc_debug, void* workspace, int* dev_err,
                           cudaStream_t stream);

int num_sms();

// Checks that the calling thread's current device is usable (sm_103) and returns
// the device address of its error word, or nullptr.
int* current_device_error_word();

// Adds n to the process-wide count of kernels enqueued by this library.
void count_launches(int n);

}  // namespace bitlinear
