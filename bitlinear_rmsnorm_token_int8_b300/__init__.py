"""BitNet b1.58 BitLinear forward on one B300 GPU (sm_103a).

Thin Python binding over the C ABI of ``libbitlinear.so`` (declared in
``include/bitlinear.h``).  Every function here only marshals arguments: it
allocates outputs with PyTorch when the caller gives none, passes raw device
pointers and the current CUDA stream, and turns a non-OK status into
:class:`BitLinearError`.  All arithmetic runs in the library's CUDA kernels;
there is no CPU fallback, and every call fails loudly if the library is missing.

Steps (page "BitNet b1.58 in Production: 1-Bit LLMs and Energy Benchmarks",
section "The Mathematical Mechanism", items 1-4):

* :func:`bitlinear_pack_weights`  absmean ternarization + 2-bit packing
* :func:`bitlinear_quant_act`     RMSNorm + per-token absmax int8 quantization
* :func:`bitlinear_forward`       exact int32 ternary contraction + dequantization
* :func:`bitlinear_linear_forward` the whole layer: the two above in one call
* :func:`bitlinear_block_forward`  the BitLinear stack of transformer layers
"""
from __future__ import annotations

import ctypes
import os

import torch

__all__ = [
    "BitLinearError", "lib", "library_path", "bitlinear_pack_weights", "bitlinear_quant_act",
    "bitlinear_forward", "bitlinear_get_device_error", "bitlinear_packed_bytes",
    "bitlinear_forward_workspace_bytes", "bitlinear_pack_workspace_bytes", "OUT_F32", "OUT_BF16",
    "STATUS", "bitlinear_kernel_launches", "bitlinear_act_ops_bytes", "FLAG_PDL", "OUT_BF16_ADD",
    "bitlinear_block_forward", "bitlinear_block_workspace_bytes", "pack_stacked", "LAYER_FIELDS",
    "bitlinear_block_trace_bytes", "block_trace_views",
    "bitlinear_linear_forward", "bitlinear_linear_workspace_bytes", "CODES_MAX_M", "bitlinear_linear_route",
    "ROUTE_FUSED", "ROUTE_CODES", "ROUTE_DECODE", "ROUTE_PREFILL", "bitlinear_prefill_cluster_size",
    "bitlinear_pack_weights_per_channel", "bitlinear_quant_act_per_tensor",
    "bitlinear_quant_act_per_tensor_workspace_bytes",
]

OUT_F32 = 0
OUT_BF16 = 1
OUT_BF16_ADD = 2
FLAG_PDL = 1
# BITLINEAR_CODES_MAX_M: bitlinear_forward given x_q contracts on the int8 codes (x_ops
# unused, no workspace) for one token, and for two whose staged codes fit in shared memory
CODES_MAX_M = 2
STATUS = {0: "OK", 1: "ERR_NULL", 2: "ERR_SHAPE", 3: "ERR_ALIGN", 4: "ERR_DTYPE", 5: "ERR_DEVICE",
          6: "ERR_CUDA", 7: "ERR_TIMEOUT", 8: "ERR_WORKSPACE", 9: "ERR_NONFINITE", 10: "ERR_FLAGS"}

_HERE = os.path.dirname(os.path.abspath(__file__))
library_path = os.path.join(_HERE, "libbitlinear.so")
_lib = None


class BitLinearError(RuntimeError):
    def __init__(self, fn: str, status: int, message: str):
        super().__init__(f"{fn}: {STATUS.get(status, status)} ({message})")
        self.status = status
        self.name = STATUS.get(status, str(status))


def lib() -> ctypes.CDLL:
    """The loaded C library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(library_path):
            raise RuntimeError(
                f"{library_path} is missing: build it with "
                "`python -m bitlinear_rmsnorm_token_int8_b300.build` (no CPU fallback exists)")
        L = ctypes.CDLL(library_path)
        P, I64, SZ, F, I = ctypes.c_void_p, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float, ctypes.c_int
        U = ctypes.c_uint
        L.bitlinear_status_string.argtypes = [I]
        L.bitlinear_status_string.restype = ctypes.c_char_p
        L.bitlinear_abi_version.restype = I
        L.bitlinear_kernel_launches.restype = ctypes.c_uint64
        L.bitlinear_packed_bytes.argtypes = [I64, I64]
        L.bitlinear_packed_bytes.restype = SZ
        L.bitlinear_pack_workspace_bytes.argtypes = [I64, I64]
        L.bitlinear_pack_workspace_bytes.restype = SZ
        L.bitlinear_pack_weights.argtypes = [P, I64, I64, F, P, P, P, P, SZ, P]
        L.bitlinear_pack_weights.restype = I
        L.bitlinear_act_ops_bytes.argtypes = [I64, I64]
        L.bitlinear_act_ops_bytes.restype = SZ
        L.bitlinear_quant_act.argtypes = [P, P, F, I64, I64, P, P, P, U, P]
        L.bitlinear_quant_act.restype = I
        L.bitlinear_pack_weights_per_channel.argtypes = [P, I64, I64, F, P, P, P]
        L.bitlinear_pack_weights_per_channel.restype = I
        L.bitlinear_quant_act_per_tensor_workspace_bytes.argtypes = [I64]
        L.bitlinear_quant_act_per_tensor_workspace_bytes.restype = SZ
        L.bitlinear_quant_act_per_tensor.argtypes = [P, I64, I64, P, P, P, P, SZ, U, P]
        L.bitlinear_quant_act_per_tensor.restype = I
        L.bitlinear_forward_workspace_bytes.argtypes = [I64, I64, I64]
        L.bitlinear_forward_workspace_bytes.restype = SZ
        L.bitlinear_forward.argtypes = [P, P, P, P, P, I64, I64, I64, I, P, P, P, SZ, P, SZ, U, P]
        L.bitlinear_forward.restype = I
        L.bitlinear_get_device_error.argtypes = [P]
        L.bitlinear_get_device_error.restype = I
        L.bitlinear_block_workspace_bytes.argtypes = [I64, I64, I64, I64]
        L.bitlinear_block_workspace_bytes.restype = SZ
        L.bitlinear_block_trace_bytes.argtypes = [I64, I64, I64, I64]
        L.bitlinear_block_trace_bytes.restype = SZ
        L.bitlinear_block_forward.argtypes = [P, I, I64, I64, I64, F, P, I64, P, SZ, P, SZ, U, P]
        L.bitlinear_block_forward.restype = I
        L.bitlinear_linear_workspace_bytes.argtypes = [I64, I64, I64]
        L.bitlinear_linear_workspace_bytes.restype = SZ
        L.bitlinear_linear_route.argtypes = [I64, I64, I64]
        L.bitlinear_linear_route.restype = I
        L.bitlinear_prefill_cluster_size.argtypes = [P, I64, I64, I64]
        L.bitlinear_prefill_cluster_size.restype = I
        L.bitlinear_linear_forward.argtypes = [P, P, F, P, P, I64, I64, I64, I, P, P, P, P, P, SZ, P, SZ, U, P]
        L.bitlinear_linear_forward.restype = I
        _lib = L
    return _lib


def _check(fn: str, status: int):
    if status != 0:
        raise BitLinearError(fn, status, lib().bitlinear_status_string(status).decode())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _prefetch(prefetch):
    """(address, bytes) of an L2 prefetch hint: None, a CUDA tensor (all of it) or a
    (tensor, bytes) pair."""
    if prefetch is None:
        return None, 0
    t, n = prefetch if isinstance(prefetch, tuple) else (prefetch, None)
    _cuda(t, "prefetch")
    total = t.numel() * t.element_size()
    return ctypes.c_void_p(t.data_ptr()), total if n is None else min(int(n), total)


def _cuda(t: torch.Tensor, name: str, dtype=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def bitlinear_kernel_launches() -> int:
    """Kernels the library has enqueued in this process so far."""
    return int(lib().bitlinear_kernel_launches())


def bitlinear_packed_bytes(N: int, K: int) -> int:
    return int(lib().bitlinear_packed_bytes(N, K))


def bitlinear_pack_workspace_bytes(N: int, K: int) -> int:
    return int(lib().bitlinear_pack_workspace_bytes(N, K))


def bitlinear_forward_workspace_bytes(M: int, N: int, K: int) -> int:
    return int(lib().bitlinear_forward_workspace_bytes(M, N, K))


def bitlinear_act_ops_bytes(M: int, K: int) -> int:
    return int(lib().bitlinear_act_ops_bytes(M, K))


def bitlinear_pack_weights(W: torch.Tensor, eps: float = 1e-5, packed=None, w_scale=None,
                           gamma=None, workspace=None, stream=None):
    """Ternarize + pack latent weights W [N,K] fp32 (CUDA).  Returns (packed, w_scale, gamma).

    ``packed`` is a flat uint8 tensor of :func:`bitlinear_packed_bytes` bytes in the
    tile-major layout (see :mod:`.layout` for the index map to the canonical [N, K/4]).
    """
    _cuda(W, "W", torch.float32)
    N, K = W.shape
    dev = W.device
    if packed is None:
        packed = torch.empty(max(bitlinear_packed_bytes(N, K), 16), dtype=torch.uint8, device=dev)
    if w_scale is None:
        w_scale = torch.empty(N, dtype=torch.float32, device=dev)
    if gamma is None:
        gamma = torch.empty(4, dtype=torch.float32, device=dev)[:1]
    if workspace is None:
        workspace = torch.empty(bitlinear_pack_workspace_bytes(N, K), dtype=torch.uint8, device=dev)
    _check("bitlinear_pack_weights", lib().bitlinear_pack_weights(
        _ptr(W), N, K, float(eps), _ptr(packed), _ptr(w_scale), _ptr(gamma), _ptr(workspace),
        workspace.numel(), _stream(stream)))
    return packed, w_scale, gamma


def bitlinear_pack_weights_per_channel(W: torch.Tensor, eps: float = 1e-5, packed=None, w_scale=None,
                                       stream=None):
    """Ternarize + pack W [N,K] fp32 (CUDA) with one absmean per output row.
    Returns (packed, w_scale) with w_scale[n] = gamma_n."""
    _cuda(W, "W", torch.float32)
    N, K = W.shape
    if packed is None:
        packed = torch.empty(max(bitlinear_packed_bytes(N, K), 16), dtype=torch.uint8, device=W.device)
    if w_scale is None:
        w_scale = torch.empty(N, dtype=torch.float32, device=W.device)
    _check("bitlinear_pack_weights_per_channel", lib().bitlinear_pack_weights_per_channel(
        _ptr(W), N, K, float(eps), _ptr(packed), _ptr(w_scale), _stream(stream)))
    return packed, w_scale


def bitlinear_quant_act_per_tensor_workspace_bytes(M: int) -> int:
    return int(lib().bitlinear_quant_act_per_tensor_workspace_bytes(M))


def bitlinear_quant_act_per_tensor(x: torch.Tensor, x_q=None, act_scale=None, x_ops=None, workspace=None,
                                   flags: int = 0, stream=None):
    """Per-tensor absmax quantization with Q_b = 128 of x [M,K] bf16 (CUDA), no RMSNorm.
    ``x_ops`` as in :func:`bitlinear_quant_act`.  Returns (x_q, act_scale[, x_ops])."""
    _cuda(x, "x", torch.bfloat16)
    M, K = x.shape
    if x_q is None:
        x_q = torch.empty((M, K), dtype=torch.int8, device=x.device)
    if act_scale is None:
        act_scale = torch.empty(max(M, 1) + 3, dtype=torch.float32, device=x.device)[:M]
    want_ops = x_ops is not None
    if x_ops is True:
        x_ops = torch.empty(max(bitlinear_act_ops_bytes(M, K), 16), dtype=torch.uint8, device=x.device)
    if workspace is None:
        workspace = torch.empty(max(bitlinear_quant_act_per_tensor_workspace_bytes(M), 256), dtype=torch.uint8,
                                device=x.device)
    _check("bitlinear_quant_act_per_tensor", lib().bitlinear_quant_act_per_tensor(
        _ptr(x), M, K, _ptr(x_q), _ptr(act_scale), _ptr(x_ops) if want_ops else None, _ptr(workspace),
        workspace.numel(), int(flags), _stream(stream)))
    return (x_q, act_scale, x_ops) if want_ops else (x_q, act_scale)


def bitlinear_quant_act(x: torch.Tensor, gain=None, rms_eps: float = 1e-5, x_q=None,
                        act_scale=None, x_ops=None, flags: int = 0, stream=None):
    """RMSNorm + per-token int8 quantization of x [M,K] bf16 (CUDA).

    ``rms_eps < 0`` skips RMSNorm; ``gain`` is the RMSNorm weight (bf16 [K]) or None.
    ``x_ops``: None (not produced), True (allocate) or a uint8 tensor of
    :func:`bitlinear_act_ops_bytes` bytes that receives the operand form of the codes.
    Returns (x_q, act_scale) or, when x_ops is requested, (x_q, act_scale, x_ops).
    """
    _cuda(x, "x", torch.bfloat16)
    M, K = x.shape
    if gain is not None:
        _cuda(gain, "gain", torch.bfloat16)
    if x_q is None:
        x_q = torch.empty((M, K), dtype=torch.int8, device=x.device)
    if act_scale is None:
        act_scale = torch.empty(max(M, 1) + 3, dtype=torch.float32, device=x.device)[:M]
    want_ops = x_ops is not None
    if x_ops is True:
        x_ops = torch.empty(max(bitlinear_act_ops_bytes(M, K), 16), dtype=torch.uint8, device=x.device)
    _check("bitlinear_quant_act", lib().bitlinear_quant_act(
        _ptr(x), _ptr(gain), float(rms_eps), M, K, _ptr(x_q), _ptr(act_scale),
        _ptr(x_ops) if want_ops else None, int(flags), _stream(stream)))
    return (x_q, act_scale, x_ops) if want_ops else (x_q, act_scale)


def bitlinear_forward(x_q, act_scale: torch.Tensor, packed: torch.Tensor,
                      w_scale: torch.Tensor, out_dtype=torch.bfloat16, y=None, acc_debug=None,
                      workspace=None, x_ops=None, flags: int = 0, K: int | None = None, stream=None,
                      prefetch=None):
    """y [M,N] = dequant(x_q . W_q^T) (CUDA).  ``acc_debug``: optional int32 [M,N] out.

    N is ``w_scale``'s length.  ``x_ops`` (from :func:`bitlinear_quant_act`) skips the
    conversion of x_q; x_q may then be None, and ``K`` must be given.  ``prefetch``: an
    L2 hint, typically the next call's packed weights (a tensor or (tensor, bytes)).
    """
    _cuda(packed, "packed", torch.uint8)
    _cuda(act_scale, "act_scale", torch.float32)
    _cuda(w_scale, "w_scale", torch.float32)
    if x_q is not None:
        _cuda(x_q, "x_q", torch.int8)
        M, K = x_q.shape
    else:
        if x_ops is None or K is None:
            raise ValueError("x_q, or x_ops and K, are required")
        M = act_scale.shape[0]
    N = w_scale.shape[0]
    if packed.numel() < bitlinear_packed_bytes(N, K):
        raise ValueError("packed is smaller than bitlinear_packed_bytes(N, K)")
    code = {torch.float32: OUT_F32, torch.bfloat16: OUT_BF16}.get(out_dtype)
    if code is None:
        raise ValueError("out_dtype must be torch.float32 or torch.bfloat16")
    if y is None:
        y = torch.empty((M, N), dtype=out_dtype, device=packed.device)
    if x_ops is None and workspace is None:
        need = bitlinear_forward_workspace_bytes(M, N, K)
        if need:
            workspace = torch.empty(need, dtype=torch.uint8, device=packed.device)
    pf, pf_bytes = _prefetch(prefetch)
    _check("bitlinear_forward", lib().bitlinear_forward(
        _ptr(x_q), _ptr(act_scale), _ptr(x_ops), _ptr(packed), _ptr(w_scale), M, N, K, code, _ptr(y),
        _ptr(acc_debug), _ptr(workspace), 0 if workspace is None else workspace.numel(),
        pf, pf_bytes, int(flags), _stream(stream)))
    return y


def bitlinear_linear_workspace_bytes(M: int, N: int, K: int) -> int:
    return int(lib().bitlinear_linear_workspace_bytes(M, N, K))


ROUTE_FUSED, ROUTE_CODES, ROUTE_DECODE, ROUTE_PREFILL = 0, 1, 2, 3


def bitlinear_linear_route(M: int, N: int, K: int) -> int:
    """Which kernels bitlinear_linear_forward runs for this shape (ROUTE_*; -1: rejected)."""
    return int(lib().bitlinear_linear_route(M, N, K))


def bitlinear_prefill_cluster_size(x_ops, M: int, N: int, K: int) -> int:
    """CTAs per cluster of the prefill contraction for operands at ``x_ops`` (a tensor or a
    raw address): 2 only for memory of the current CUDA device; -1 off the prefill route."""
    addr = x_ops.data_ptr() if isinstance(x_ops, torch.Tensor) else x_ops
    return int(lib().bitlinear_prefill_cluster_size(ctypes.c_void_p(addr), M, N, K))


def bitlinear_linear_forward(x: torch.Tensor, gain, rms_eps: float, packed: torch.Tensor,
                             w_scale: torch.Tensor, out_dtype=torch.bfloat16, y=None, x_q=None,
                             act_scale=None, acc_debug=None, workspace=None, flags: int = 0,
                             residual: bool = False, stream=None, prefetch=None):
    """The BitLinear layer: y [M,N] = dequant(quant(RMSNorm(x)) . W_q^T) from bf16 x [M,K] (CUDA).

    ``gain``: RMSNorm weight (bf16 [K]) or None; ``rms_eps < 0`` skips RMSNorm.  ``x_q``
    (int8 [M,K]) and ``act_scale`` (fp32 [M]) receive the codes and scales when given.
    ``residual``: y (bf16) holds the residual on entry and receives y + result.
    One token with K <= 8192 (K <= 16384 for at least 12 MiB of packed weights) runs as a
    single kernel; :func:`bitlinear_linear_route`
    tells which kernels a shape takes (the results are the same on every route).
    ``prefetch``: an L2 hint, typically the next call's packed weights (see
    :func:`bitlinear_forward`).
    """
    _cuda(x, "x", torch.bfloat16)
    _cuda(packed, "packed", torch.uint8)
    _cuda(w_scale, "w_scale", torch.float32)
    if gain is not None:
        _cuda(gain, "gain", torch.bfloat16)
    M, K = x.shape
    N = w_scale.shape[0]
    if packed.numel() < bitlinear_packed_bytes(N, K):
        raise ValueError("packed is smaller than bitlinear_packed_bytes(N, K)")
    code = {torch.float32: OUT_F32, torch.bfloat16: OUT_BF16}.get(out_dtype)
    if code is None:
        raise ValueError("out_dtype must be torch.float32 or torch.bfloat16")
    if residual:
        if y is None or out_dtype != torch.bfloat16:
            raise ValueError("residual needs a bf16 y")
        code = OUT_BF16_ADD
    if y is None:
        y = torch.empty((M, N), dtype=out_dtype, device=x.device)
    if workspace is None:
        need = bitlinear_linear_workspace_bytes(M, N, K)
        workspace = torch.empty(need, dtype=torch.uint8, device=x.device) if need else None
    _check("bitlinear_linear_forward", lib().bitlinear_linear_forward(
        _ptr(x), _ptr(gain), float(rms_eps), _ptr(packed), _ptr(w_scale), M, N, K, code, _ptr(y),
        _ptr(x_q), _ptr(act_scale), _ptr(acc_debug), _ptr(workspace),
        0 if workspace is None else workspace.numel(), *_prefetch(prefetch), int(flags), _stream(stream)))
    return y


LAYER_FIELDS = ("qkv", "qkv_scale", "o", "o_scale", "gate_up", "gate_up_scale", "down", "down_scale",
                "gain_qkv", "gain_o", "gain_gate_up", "gain_down")


class _Layer(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in LAYER_FIELDS]


def pack_stacked(Ws, eps: float = 1e-5, stream=None):
    """Packs several latent matrices (each [N_i, K] fp32 CUDA) as one stacked projection:
    each keeps its own gamma.  Every N_i but the last must be a multiple of 128 (the
    packed layout's row tile), the last a multiple of 16.  Returns (packed, w_scale)."""
    for i, W in enumerate(Ws):
        n = W.shape[0]
        if n % 16 != 0 or (i + 1 < len(Ws) and n % 128 != 0):
            raise ValueError("stacked matrices need N_i % 128 == 0 (the last: N % 16 == 0)")
    parts = [bitlinear_pack_weights(W, eps, stream=stream)[:2] for W in Ws]
    return torch.cat([p for p, _ in parts]), torch.cat([s for _, s in parts])


def bitlinear_block_workspace_bytes(M: int, H: int, NQKV: int, F: int) -> int:
    return int(lib().bitlinear_block_workspace_bytes(M, H, NQKV, F))


def bitlinear_block_trace_bytes(M: int, H: int, NQKV: int, F: int) -> int:
    return int(lib().bitlinear_block_trace_bytes(M, H, NQKV, F))


def block_trace_views(trace: torch.Tensor, layer: int, M: int, H: int, NQKV: int, F: int) -> dict:
    """Views of one layer's part of a bitlinear_block_forward trace (the layout that
    bitlinear_block_trace_bytes documents): xq_{qkv,o,gate_up,down} int8,
    sc_{...} fp32, qkv bf16, x_mid bf16, gate_up fp32, x_out bf16."""
    stride = bitlinear_block_trace_bytes(M, H, NQKV, F)
    base = trace[layer * stride:(layer + 1) * stride]
    out, off = {}, 0

    def take(name, nbytes, dtype, shape):
        nonlocal off
        out[name] = base[off:off + nbytes].view(dtype).view(*shape)
        off = (off + nbytes + 255) // 256 * 256

    for name, k in (("qkv", H), ("o", H), ("gate_up", H), ("down", F)):
        take("xq_" + name, M * k, torch.int8, (M, k))
    for name in ("qkv", "o", "gate_up", "down"):
        take("sc_" + name, 4 * M, torch.float32, (M,))
    take("qkv", 2 * M * NQKV, torch.bfloat16, (M, NQKV))
    take("x_mid", 2 * M * H, torch.bfloat16, (M, H))
    take("gate_up", 8 * M * F, torch.float32, (M, 2 * F))
    take("x_out", 2 * M * H, torch.bfloat16, (M, H))
    return out


def bitlinear_block_forward(layers, x: torch.Tensor, H: int, NQKV: int, F: int, rms_eps: float = 1e-5,
                            workspace=None, flags: int = 0, stream=None, trace=None):
    """The BitLinear stack of len(layers) transformer layers on x [M, H] bf16 (CUDA), in place.

    ``layers``: dicts with the CUDA tensors named in :data:`LAYER_FIELDS` (packed weights,
    fp32 per-row scales, bf16 RMSNorm gains).  ``trace``: None, or a uint8 CUDA tensor of
    len(layers) * :func:`bitlinear_block_trace_bytes` bytes (256-byte aligned) that
    receives every layer's intermediates (read them with :func:`block_trace_views`).
    Returns x.
    """
    _cuda(x, "x", torch.bfloat16)
    M = x.shape[0]
    arr = (_Layer * max(len(layers), 1))()
    for i, layer in enumerate(layers):
        for n in LAYER_FIELDS:
            t = layer[n]
            _cuda(t, n)
            setattr(arr[i], n, t.data_ptr())
    if workspace is None:
        workspace = torch.empty(bitlinear_block_workspace_bytes(M, H, NQKV, F) + 256, dtype=torch.uint8,
                                device=x.device)
    if trace is not None:
        _cuda(trace, "trace", torch.uint8)
    _check("bitlinear_block_forward", lib().bitlinear_block_forward(
        ctypes.cast(arr, ctypes.c_void_p), len(layers), H, NQKV, F, float(rms_eps), _ptr(x), M,
        _ptr(workspace), workspace.numel(), _ptr(trace), 0 if trace is None else trace.numel(), int(flags),
        _stream(stream)))
    return x


def bitlinear_get_device_error(stream=None) -> int:
    """Waits for the stream; returns and clears the device error word (0 = none)."""
    return int(lib().bitlinear_get_device_error(_stream(stream)))
