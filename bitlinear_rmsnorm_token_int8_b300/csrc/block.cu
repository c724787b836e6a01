// bitlinear_block_forward: the BitLinear projections of a stack of BitNet
// b1.58 transformer layers, chained on one stream (contract in bitlinear.h).
//
// Per layer eight kernels (five for one token, where the QKV, O and gate+up
// layers each run as one kernel that also quantizes), each launched as a
// programmatic dependent of the previous one (its weights are read before the
// previous kernel ends):
//   quant(x, g_qkv) -> forward(qkv, bf16) -> quant(qkv[:, :H], g_o)
//   -> forward(o, bf16 residual add into x) -> quant(x, g_gate_up)
//   -> forward(gate_up, fp32) -> quant(ReLU^2-gated h, g_down)
//   -> forward(down, bf16 residual add into x).
// The ReLU^2 gating is fused into the quantization of h (it reads the fp32
// gate and up rows), the residual adds into the contraction epilogues.  Every
// contraction pulls the packed weights of the projection after it into L2.
//
// With a trace buffer the kernels also leave, per layer, every BitLinear's
// int8 codes and scales and the intermediate tensors there (four small copy
// kernels per layer add the qkv, residual and gate+up tensors), so that each
// BitLinear can be checked against a reference fed its exact input.
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/bitlinear.h"
#include "act_ops.cuh"
#include "device_util.cuh"
#include "internal.h"

namespace bitlinear {
namespace {

inline size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

struct BlockWs {
  uint8_t* ops;      // operand planes, largest K
  float* scale;      // act_scale [M]
  uint16_t* qkv;     // bf16 [M, NQKV]
  float* gu;         // fp32 [M, 2F]
  size_t bytes;
};

BlockWs block_ws(uint8_t* base, int64_t M, int64_t H, int64_t NQKV, int64_t F) {
  BlockWs w;
  const int64_t kmax = H > F ? H : F;
  size_t off = 0;
  w.ops = base + off;
  off = align256(off + act_ops_bytes(M, kmax));
  w.scale = reinterpret_cast<float*>(base + off);
  off = align256(off + (size_t)M * 4);
  w.qkv = reinterpret_cast<uint16_t*>(base + off);
  off = align256(off + (size_t)M * NQKV * 2);
  w.gu = reinterpret_cast<float*>(base + off);
  off = align256(off + (size_t)M * 2 * F * 4);
  w.bytes = off;
  return w;
}

// One layer's trace, in this order (each part 256-byte aligned): the codes of the
// four BitLinears' inputs (qkv, o, gate_up: [M, H]; down: [M, F] int8), their
// scales ([4][M] fp32), qkv ([M, NQKV] bf16), x after the O residual ([M, H] bf16),
// gate|up ([M, 2F] fp32), x after the down residual ([M, H] bf16).
struct BlockTrace {
  int8_t* xq[4];
  float* sc[4];
  uint16_t* qkv;
  uint16_t* x_mid;
  float* gu;
  uint16_t* x_out;
  size_t bytes;
};

BlockTrace block_trace(uint8_t* base, int64_t M, int64_t H, int64_t NQKV, int64_t F) {
  BlockTrace t;
  size_t off = 0;
  for (int b = 0; b < 4; ++b) {
    t.xq[b] = reinterpret_cast<int8_t*>(base + off);
    off = align256(off + (size_t)M * (b == 3 ? F : H));
  }
  for (int b = 0; b < 4; ++b) {
    t.sc[b] = reinterpret_cast<float*>(base + off);
    off = align256(off + (size_t)M * 4);
  }
  t.qkv = reinterpret_cast<uint16_t*>(base + off);
  off = align256(off + (size_t)M * NQKV * 2);
  t.x_mid = reinterpret_cast<uint16_t*>(base + off);
  off = align256(off + (size_t)M * H * 2);
  t.gu = reinterpret_cast<float*>(base + off);
  off = align256(off + (size_t)M * 2 * F * 4);
  t.x_out = reinterpret_cast<uint16_t*>(base + off);
  off = align256(off + (size_t)M * H * 2);
  t.bytes = off;
  return t;
}

// dst = src, 16 bytes per thread step, after the previous kernel (programmatic
// dependent launch: it starts early and waits for the data).
__global__ void trace_copy_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst, int64_t n16) {
  pdl_launch_dependents();
  pdl_wait();
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n16; i += (int64_t)gridDim.x * blockDim.x)
    dst[i] = __ldcg(src + i);
}

cudaError_t launch_trace_copy(const void* src, void* dst, size_t bytes, cudaStream_t stream) {
  const int64_t n16 = (int64_t)(bytes / 16);
  int64_t blocks = (n16 + 255) / 256;
  const int64_t cap = (int64_t)num_sms() * 4;
  if (blocks > cap) blocks = cap;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(blocks > 0 ? blocks : 1), 1, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, trace_copy_kernel, static_cast<const uint4*>(src), static_cast<uint4*>(dst),
                                     n16);
  count_launches(1);
  return e;
}

}  // namespace
}  // namespace bitlinear

using namespace bitlinear;

extern "C" size_t bitlinear_block_workspace_bytes(int64_t M, int64_t H, int64_t NQKV, int64_t F) {
  if (M < 1 || H < 1 || NQKV < 1 || F < 1) return 0;
  return block_ws(nullptr, M, H, NQKV, F).bytes;
}

extern "C" size_t bitlinear_block_trace_bytes(int64_t M, int64_t H, int64_t NQKV, int64_t F) {
  if (M < 1 || H < 1 || NQKV < 1 || F < 1) return 0;
  return block_trace(nullptr, M, H, NQKV, F).bytes;
}

extern "C" bitlinear_status bitlinear_block_forward(const bitlinear_layer* layers, int n_layers,
                                                    int64_t H, int64_t NQKV, int64_t F, float rms_eps,
                                                    void* x_bf16, int64_t M, void* workspace,
                                                    size_t workspace_bytes, void* trace, size_t trace_bytes,
                                                    unsigned flags, void* stream) {
  if (n_layers < 0 || M < 1 || M > (int64_t(1) << 20) || H < 128 || H % 128 != 0 || H > 65536 ||
      F < 128 || F % 128 != 0 || F > 65536 || NQKV < H || NQKV % 16 != 0 || NQKV > (int64_t(1) << 24) ||
      !(rms_eps >= 0.0f))
    return BITLINEAR_ERR_SHAPE;
  if (flags & ~BITLINEAR_FLAG_PDL) return BITLINEAR_ERR_FLAGS;
  if (n_layers == 0) return BITLINEAR_OK;
  if (!layers || !x_bf16 || !workspace) return BITLINEAR_ERR_NULL;
  if ((reinterpret_cast<uintptr_t>(x_bf16) & 15) || (reinterpret_cast<uintptr_t>(workspace) & 255) ||
      (reinterpret_cast<uintptr_t>(trace) & 255))
    return BITLINEAR_ERR_ALIGN;
  if (workspace_bytes < bitlinear_block_workspace_bytes(M, H, NQKV, F)) return BITLINEAR_ERR_WORKSPACE;
  const size_t tstride = trace ? bitlinear_block_trace_bytes(M, H, NQKV, F) : 0;
  if (trace && trace_bytes < tstride * (size_t)n_layers) return BITLINEAR_ERR_WORKSPACE;
  for (int l = 0; l < n_layers; ++l) {
    const bitlinear_layer& L = layers[l];
    const void* ptrs[12] = {L.qkv, L.qkv_scale, L.o, L.o_scale, L.gate_up, L.gate_up_scale, L.down,
                            L.down_scale, L.gain_qkv, L.gain_o, L.gain_gate_up, L.gain_down};
    for (const void* q : ptrs) {
      if (!q) return BITLINEAR_ERR_NULL;
      if (reinterpret_cast<uintptr_t>(q) & 15) return BITLINEAR_ERR_ALIGN;
    }
  }
  int* err = current_device_error_word();
  if (!err) return BITLINEAR_ERR_DEVICE;
  const BlockWs w = block_ws(static_cast<uint8_t*>(workspace), M, H, NQKV, F);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const uint16_t* x = static_cast<const uint16_t*>(x_bf16);
  bool pdl = (flags & BITLINEAR_FLAG_PDL) != 0;
  cudaError_t e = cudaSuccess;
  BlockTrace tr = {};                        // this layer's trace (when tracing)
  // Per projection: int8 codes for the CUDA-core contraction (one or two tokens) or
  // the tensor-core operand form, and the token scales: in the workspace, or, when
  // tracing, the codes and scales go to the trace (the contraction reads them there).
  auto codes_of = [&](int b) { return trace ? tr.xq[b] : reinterpret_cast<int8_t*>(w.ops); };
  auto scale_of = [&](int b) { return trace ? tr.sc[b] : w.scale; };
  auto quant = [&](int b, const uint16_t* in, int64_t ld, const float* glu, const void* gain, int64_t N, int64_t K) {
    const bool codes = codes_route(M, N, K);
    if (e == cudaSuccess)
      e = launch_quant_act_ex(in, ld, glu, static_cast<const uint16_t*>(gain), rms_eps, M, K,
                              (codes || trace) ? codes_of(b) : nullptr, scale_of(b), codes ? nullptr : w.ops, pdl,
                              s);
    pdl = true;                         // everything after the first kernel is ours
  };
  auto forward = [&](int b, const uint8_t* packed, const float* wscale, int64_t N, int64_t K, int out_dtype, void* y,
                     L2Prefetch next) {
    const bool codes = codes_route(M, N, K);
    if (e == cudaSuccess)
      e = launch_forward(codes ? codes_of(b) : nullptr, scale_of(b), codes ? nullptr : w.ops, packed, wscale, M, N,
                         K, out_dtype, y, nullptr, nullptr, err, true, s, next);
  };
  auto weights = [](const uint8_t* packed, int64_t N, int64_t K) {
    L2Prefetch pf;
    pf.p = packed;
    pf.bytes = (uint64_t)packed_layout_bytes(N, K);
    return pf;
  };
  // one projection on bf16 rows `in` (pitch ld): for one token one kernel (RMSNorm,
  // quantization and contraction together), else quantization, then the contraction
  auto layer = [&](int b, const uint16_t* in, int64_t ld, const void* gain, const uint8_t* packed,
                   const float* wscale, int64_t N, int64_t K, int out_dtype, void* y, L2Prefetch next) {
    if (fused_route(M, N, K)) {              // one token: the row pitch does not matter
      if (e == cudaSuccess)
        e = launch_layer_cc(in, static_cast<const uint16_t*>(gain), rms_eps, packed, wscale, M, N, K, out_dtype, y,
                            trace ? tr.xq[b] : nullptr, trace ? tr.sc[b] : nullptr, nullptr, pdl, s, next);
      pdl = true;
      return;
    }
    quant(b, in, ld, nullptr, gain, N, K);
    forward(b, packed, wscale, N, K, out_dtype, y, next);
  };
  auto keep = [&](const void* src, void* dst, size_t bytes) {
    if (trace && e == cudaSuccess) e = launch_trace_copy(src, dst, bytes, s);
  };
  for (int l = 0; l < n_layers && e == cudaSuccess; ++l) {
    const bitlinear_layer& L = layers[l];
    if (trace) tr = block_trace(static_cast<uint8_t*>(trace) + (size_t)l * tstride, M, H, NQKV, F);
    const L2Prefetch w_o = weights(L.o, H, H), w_gu = weights(L.gate_up, 2 * F, H), w_down = weights(L.down, H, F);
    const L2Prefetch w_next = l + 1 < n_layers ? weights(layers[l + 1].qkv, NQKV, H) : L2Prefetch{};
    layer(0, x, H, L.gain_qkv, L.qkv, L.qkv_scale, NQKV, H, BITLINEAR_OUT_BF16, w.qkv, w_o);
    keep(w.qkv, tr.qkv, (size_t)M * NQKV * 2);
    // the query slice stands in for attention
    layer(1, w.qkv, NQKV, L.gain_o, L.o, L.o_scale, H, H, BITLINEAR_OUT_BF16_ADD, x_bf16, w_gu);
    keep(x_bf16, tr.x_mid, (size_t)M * H * 2);
    layer(2, x, H, L.gain_gate_up, L.gate_up, L.gate_up_scale, 2 * F, H, BITLINEAR_OUT_F32, w.gu, w_down);
    keep(w.gu, tr.gu, (size_t)M * 2 * F * 4);
    quant(3, nullptr, F, w.gu, L.gain_down, H, F);               // h = bf16(relu(gate)^2 * up)
    forward(3, L.down, L.down_scale, H, F, BITLINEAR_OUT_BF16_ADD, x_bf16, w_next);
    keep(x_bf16, tr.x_out, (size_t)M * H * 2);
  }
  return e == cudaSuccess ? BITLINEAR_OK : BITLINEAR_ERR_CUDA;
}
