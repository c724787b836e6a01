// Host-side declarations shared by the translation units of libbitlinear.
// Launchers validate nothing: api.cu checks every argument before calling them.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace bitlinear {

// Device status values written into the per-device error word (same numbers
// as the public bitlinear_status codes).
constexpr int kDevErrTimeout = 7;
constexpr int kDevErrNonFinite = 9;

// ---- packed weight layout -------------------------------------------------
// Tile-major and pre-swizzled for the contraction kernels: rows padded to
// Np = N rounded up to 16 and grouped in tiles of 128 (the last tile holds the
// remaining Np % 128 rows, if any), K in segments of 512 (padded with zero
// codes), 128 bytes per row and segment.  Tiles follow one another; within a
// tile of R rows, segment s is one contiguous block of R x 128 bytes, in which
// the 16-byte chunk c of row r sits at chunk position c ^ (r % 8).  So the
// weights of any run of segments of one tile are one contiguous range, which
// one bulk copy moves.  Byte b of row n's canonical packed row (b = k / 4):
//   (n / 128) * 128 * nseg * 128 + (b / 128) * R * 128 + (n % 128) * 128
//     + (((b % 128) / 16) ^ (n % 8)) * 16 + b % 16,   R = min(128, Np - 128 (n / 128)).
constexpr int64_t kSegK = 512;
constexpr int64_t kTileRows = 128;
inline int64_t packed_nseg(int64_t K) { return (K + kSegK - 1) / kSegK; }
inline int64_t packed_rows(int64_t N) { return (N + 15) / 16 * 16; }
inline int64_t packed_layout_bytes(int64_t N, int64_t K) { return packed_rows(N) * packed_nseg(K) * 128; }

// A device range that a call's kernels ask the copy engine to pull into L2 while
// they run (typically the packed weights of the call that follows on the stream).
// It is only a cache hint: nothing reads it into registers or shared memory, and
// L2 is the point of coherence, so it can never make a kernel see stale data.
struct L2Prefetch {
  const uint8_t* p = nullptr;
  uint64_t bytes = 0;
};

// ---- pack_weights --------------------------------------------------------
// Workspace layout (bytes): [0, 2048) 256 uint64 exponent bins of sum|W|,
// [2048, 2056) gamma and d = fl32(gamma + eps) as two floats.
constexpr size_t kPackBinsBytes = 256 * sizeof(unsigned long long);
constexpr size_t kPackWorkspaceBytes = kPackBinsBytes + 16;

cudaError_t launch_pack_weights(const float* W, int64_t N, int64_t K, float eps, uint8_t* packed,
                                float* w_scale, float* gamma_out, void* workspace, int* dev_err,
                                cudaStream_t stream);

// The same packing with one absmean per output row (written to w_scale); no scratch.
cudaError_t launch_pack_weights_per_channel(const float* W, int64_t N, int64_t K, float eps, uint8_t* packed,
                                            float* w_scale, int* dev_err, cudaStream_t stream);

// Per-tensor absmax quantization with Q_b = 128 (no RMSNorm): per-row maxima into
// `row_max` (M floats of scratch), then codes with one scale for all rows.
cudaError_t launch_quant_act_per_tensor(const uint16_t* x, int64_t M, int64_t K, int8_t* x_q, float* act_scale,
                                        uint8_t* x_ops, float* row_max, bool pdl, cudaStream_t stream);

// ---- quant_act -----------------------------------------------------------
// x_ops: optional tensor-core operand planes of the codes (act_ops.cuh), or nullptr.
cudaError_t launch_quant_act(const uint16_t* x, const uint16_t* gain, float rms_eps, int64_t M,
                             int64_t K, int8_t* x_q, float* act_scale, uint8_t* x_ops, bool pdl,
                             cudaStream_t stream);

// Same with a row pitch `ld` (elements, a multiple of 8) or, if `glu` is set, the
// ReLU^2-gated rows of fp32 [gate | up] (x unused).  x_q may be null.
cudaError_t launch_quant_act_ex(const uint16_t* x, int64_t ld, const float* glu, const uint16_t* gain,
                                float rms_eps, int64_t M, int64_t K, int8_t* x_q, float* act_scale,
                                uint8_t* x_ops, bool pdl, cudaStream_t stream);

// ---- activation operands ---------------------------------------------------
size_t act_ops_bytes(int64_t M, int64_t K);
cudaError_t launch_act_ops_from_codes(const int8_t* x_q, int64_t M, int64_t K, uint8_t* ops,
                                      bool pdl, cudaStream_t stream);

// ---- forward ---------------------------------------------------------------
size_t forward_workspace_bytes(int64_t M, int64_t N, int64_t K);

// x_ops may be nullptr: the operands are then derived from x_q into the workspace.
cudaError_t launch_forward(const int8_t* x_q, const float* act_scale, const uint8_t* x_ops,
                           const uint8_t* packed, const float* w_scale, int64_t M, int64_t N,
                           int64_t K, int out_dtype, void* y, int32_t* acc_debug, void* workspace,
                           int* dev_err, bool pdl, cudaStream_t stream, L2Prefetch pf = {});

// Decode contraction (M <= kDecodeMaxM) on tcgen05: launch plan and launcher.
struct DecodePlan {
  int Mt;            // tokens padded to 8 (MMA n = 2 Mt: both operand planes)
  int nseg;          // 512-wide K segments
  int ntile;         // 128-row weight tiles
  int S;             // K slices = CTAs per cluster
  int G;             // segments per pipeline stage
  int NS;            // pipeline stages
  int stage_bytes;   // shared bytes per stage (weights, then operands)
  int64_t smem;      // dynamic shared memory per CTA
};
DecodePlan decode_plan(int64_t M, int64_t N, int64_t K, int sms);
bool decode_plan_ok(const DecodePlan& pl);

cudaError_t launch_decode_tc(const uint8_t* x_ops, const float* act_scale, const uint8_t* packed,
                             const float* w_scale, int64_t M, int64_t N, int64_t K, int out_dtype,
                             void* y, int32_t* acc_debug, int* dev_err, bool pdl,
                             cudaStream_t stream, L2Prefetch pf = {});

// Decode contraction for one or two tokens on the CUDA cores (int8 dot products,
// one persistent CTA per SM), reading the int8 codes x_q; shared memory per CTA
// from decode_cc_smem (0: the shape does not fit).
constexpr int64_t kCodesMaxM = 2;
size_t decode_cc_smem(int64_t M, int64_t K);
// True when bitlinear_forward with x_q takes that kernel: 1 <= M <= kCodesMaxM and
// the tokens' staged codes and the weight ring fit in shared memory.
bool codes_route(int64_t M, int64_t N, int64_t K);
cudaError_t launch_codes_cc(const int8_t* x_q, const float* act_scale, const uint8_t* packed,
                            const float* w_scale, int64_t M, int64_t N, int64_t K, int out_dtype,
                            void* y, int32_t* acc_debug, bool pdl, cudaStream_t stream,
                            L2Prefetch pf = {});

// The whole layer (RMSNorm + quantization + contraction) for one token in one kernel,
// when the codes route applies and K <= 8192 (K <= 16384 for matrices of at least
// kCcMinBytes); x_q and act_scale outputs optional.
bool fused_route(int64_t M, int64_t N, int64_t K);
cudaError_t launch_layer_cc(const uint16_t* x, const uint16_t* gain, float rms_eps, const uint8_t* packed,
                            const float* w_scale, int64_t M, int64_t N, int64_t K, int out_dtype, void* y,
                            int8_t* x_q, float* act_scale, int32_t* acc_debug, bool pdl, cudaStream_t stream,
                            L2Prefetch pf = {});

// The CUDA-core kernels of many small CTAs (decode_dp4a.cu), which launch_codes_cc
// and launch_layer_cc take for matrices below kCcMinBytes of packed weights: there
// they finish sooner in a chain of dependent launches than the persistent kernel.
constexpr int64_t kCcMinBytes = int64_t(12) << 20;
bool dp4a_codes_ok(int64_t M, int64_t N, int64_t K);
bool dp4a_layer_ok(int64_t M, int64_t N, int64_t K);
cudaError_t launch_decode_dp4a(const int8_t* x_q, const float* act_scale, const uint8_t* packed,
                               const float* w_scale, int64_t M, int64_t N, int64_t K, int out_dtype,
                               void* y, int32_t* acc_debug, bool pdl, cudaStream_t stream, L2Prefetch pf);
cudaError_t launch_linear_dp4a(const uint16_t* x, const uint16_t* gain, float rms_eps, const uint8_t* packed,
                               const float* w_scale, int64_t N, int64_t K, int out_dtype, void* y, int8_t* x_q,
                               float* act_scale, int32_t* acc_debug, bool pdl, cudaStream_t stream,
                               L2Prefetch pf);

int num_sms();

// ---- tensor maps and the prefill contraction ---------------------------------

// CTAs per cluster of the prefill contraction for operands at x_ops (2 only when
// x_ops is memory of the current device and N spans two weight blocks), and tokens
// per tile (256, or 128 when that fills more SMs) for that cluster size.
int prefill_cluster(const void* x_ops, int64_t N);
int prefill_tile_tokens(int64_t M, int64_t N, int CL, int sms);

cudaError_t launch_prefill_tc(const uint8_t* x_ops, const float* act_scale, const uint8_t* packed,
                              const float* w_scale, int64_t M, int64_t N, int64_t K, int out_dtype,
                              void* y, int32_t* acc_debug, int* dev_err, bool pdl,
                              cudaStream_t stream);



// Checks that the calling thread's current device is usable (sm_103) and returns
// the device address of its error word, or nullptr.
int* current_device_error_word();

// Adds n to the process-wide count of kernels enqueued by this library.
void count_launches(int n);

}  // namespace bitlinear
