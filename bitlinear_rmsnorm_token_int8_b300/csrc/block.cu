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
// gate and up rows), the residual adds into the contraction epilogues.
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/bitlinear.h"
#include "act_ops.cuh"
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

}  // namespace
}  // namespace bitlinear

using namespace bitlinear;

extern "C" size_t bitlinear_block_workspace_bytes(int64_t M, int64_t H, int64_t NQKV, int64_t F) {
  if (M < 1 || H < 1 || NQKV < 1 || F < 1) return 0;
  return block_ws(nullptr, M, H, NQKV, F).bytes;
}

extern "C" bitlinear_status bitlinear_block_forward(const bitlinear_layer* layers, int n_layers,
                                                    int64_t H, int64_t NQKV, int64_t F, float rms_eps,
                                                    void* x_bf16, int64_t M, void* workspace,
                                                    size_t workspace_bytes, unsigned flags, void* stream) {
  if (n_layers < 0 || M < 1 || M > (int64_t(1) << 20) || H < 128 || H % 128 != 0 || H > 65536 ||
      F < 128 || F % 128 != 0 || F > 65536 || NQKV < H || NQKV % 16 != 0 || NQKV > (int64_t(1) << 24) ||
      !(rms_eps >= 0.0f))
    return BITLINEAR_ERR_SHAPE;
  if (flags & ~BITLINEAR_FLAG_PDL) return BITLINEAR_ERR_FLAGS;
  if (n_layers == 0) return BITLINEAR_OK;
  if (!layers || !x_bf16 || !workspace) return BITLINEAR_ERR_NULL;
  if ((reinterpret_cast<uintptr_t>(x_bf16) & 15) || (reinterpret_cast<uintptr_t>(workspace) & 255))
    return BITLINEAR_ERR_ALIGN;
  if (workspace_bytes < bitlinear_block_workspace_bytes(M, H, NQKV, F)) return BITLINEAR_ERR_WORKSPACE;
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
  // per projection: int8 codes in the operand region for the CUDA-core contraction
  // (one or two tokens), or the tensor-core operand form.  Every contraction pulls
  // the packed weights of the projection after it into L2 while it runs, so the
  // weight stream continues across the launches; the first quantization pulls in
  // the first projection's.
  int8_t* const codes_buf = reinterpret_cast<int8_t*>(w.ops);
  auto quant = [&](const uint16_t* in, int64_t ld, const float* glu, const void* gain, int64_t N, int64_t K,
                   L2Prefetch pf) {
    const bool codes = codes_route(M, N, K);
    if (e == cudaSuccess)
      e = launch_quant_act_ex(in, ld, glu, static_cast<const uint16_t*>(gain), rms_eps, M, K,
                              codes ? codes_buf : nullptr, w.scale, codes ? nullptr : w.ops, pdl, s, pf);
    pdl = true;                         // everything after the first kernel is ours
  };
  auto forward = [&](const uint8_t* packed, const float* wscale, int64_t N, int64_t K, int out_dtype, void* y,
                     L2Prefetch next) {
    const bool codes = codes_route(M, N, K);
    if (e == cudaSuccess)
      e = launch_forward(codes ? codes_buf : nullptr, w.scale, codes ? nullptr : w.ops, packed, wscale, M, N, K,
                         out_dtype, y, nullptr, nullptr, err, true, s, next);
  };
  auto weights = [](const uint8_t* packed, int64_t N, int64_t K) {
    L2Prefetch pf;
    pf.p = packed;
    pf.bytes = (uint64_t)packed_layout_bytes(N, K);
    return pf;
  };
  // one projection on bf16 rows `in` (pitch ld): for one token one kernel (RMSNorm,
  // quantization and contraction together), else quantization, then the contraction
  auto layer = [&](const uint16_t* in, int64_t ld, const void* gain, const uint8_t* packed, const float* wscale,
                   int64_t N, int64_t K, int out_dtype, void* y, L2Prefetch own, L2Prefetch next) {
    if (fused_route(M, N, K)) {
      if (e == cudaSuccess)
        e = launch_layer_cc(in, static_cast<const uint16_t*>(gain), rms_eps, packed, wscale, M, N, K, out_dtype, y,
                            nullptr, nullptr, nullptr, pdl, s, next);
      pdl = true;
      return;
    }
    quant(in, ld, nullptr, gain, N, K, own);
    forward(packed, wscale, N, K, out_dtype, y, next);
  };
  for (int l = 0; l < n_layers && e == cudaSuccess; ++l) {
    const bitlinear_layer& L = layers[l];
    const L2Prefetch w_o = weights(L.o, H, H), w_gu = weights(L.gate_up, 2 * F, H), w_down = weights(L.down, H, F);
    const L2Prefetch w_next = l + 1 < n_layers ? weights(layers[l + 1].qkv, NQKV, H) : L2Prefetch{};
    layer(x, H, L.gain_qkv, L.qkv, L.qkv_scale, NQKV, H, BITLINEAR_OUT_BF16, w.qkv,
          l == 0 ? weights(L.qkv, NQKV, H) : L2Prefetch{}, w_o);
    // the query slice stands in for attention
    layer(w.qkv, NQKV, L.gain_o, L.o, L.o_scale, H, H, BITLINEAR_OUT_BF16_ADD, x_bf16, L2Prefetch{}, w_gu);
    layer(x, H, L.gain_gate_up, L.gate_up, L.gate_up_scale, 2 * F, H, BITLINEAR_OUT_F32, w.gu, L2Prefetch{}, w_down);
    quant(nullptr, F, w.gu, L.gain_down, H, F, L2Prefetch{});     // h = bf16(relu(gate)^2 * up)
    forward(L.down, L.down_scale, H, F, BITLINEAR_OUT_BF16_ADD, x_bf16, w_next);
  }
  return e == cudaSuccess ? BITLINEAR_OK : BITLINEAR_ERR_CUDA;
}
