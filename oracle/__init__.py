"""CPU oracle for the BitNet b1.58 BitLinear forward.

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference leg of ``bench.py`` may import this package.  The CUDA
library never links, loads or calls it, and this package imports nothing from
the CUDA package: the two share no code.  Inputs are numpy arrays; bf16 values
travel as their raw ``uint16`` bit patterns.

The arithmetic lives in ``bitlinear_oracle.c`` (plain single-threaded C, built
with ``build()``); this module adds the exact rational rounding of the absmean
and the composition of the steps.  Each function names the passage it follows:

* [P4-eq]   "BitNet b1.58 in Production: 1-Bit LLMs and Energy Benchmarks",
            section "The Mathematical Mechanism: BitLinear vs Standard Linear",
            items 1-4.
* [P4-code] same page, "Production Multi-File Implementation", bit_linear.py.
* [P5-lut]  "BitNet 1-bit LLM Inference Framework", section "How the LUT Kernel
            Works".
* [P5-mask] same page, section "The Difference in How Computation Works"
            (mask form: y = (W==1) x - (W==-1) x).

* [P5-block] "BitNet 1-bit LLM Inference Framework", section "A Full BitNet
            Transformer Block" (q/k/v/o and gate/up/down projections, residual
            adds around the attention and the FFN).
* [P5-aq]   same page, BitLinear.activation_quantize (per-tensor scale, Q_b = 128).
* [P2-wr]   "BitNet-2B-4T: Inside the 2B-Parameter, 4T-Token 1-Bit LLM", section
            "Weight Representation: Ternary + Scale, Not Pure Binary"
            (per-output-channel scaling W_bit x s, s in R^d).

Parity pins: every function here is pinned by ``tests/test_oracle.py`` (hand-worked
values in ``tests/golden/worked_examples.json``, including the bf16 rounding of
``f32_to_bf16_bits`` and the clamp of tiny rows);
``block_layer`` is pinned only by identities (zero projections leave the
residual stream unchanged, the gate's closed form) and by a recomputation
with dense fp64 matmuls, its attention stand-in being a reading, not a
definition (see the function's docstring).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from fractions import Fraction

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "bitlinear_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None

EPS_W = np.float32(1e-5)      # weight eps of Clip(Round(W/(gamma+eps)))
QB = 127                      # Q_b = 2^(8-1) - 1 for 8-bit activations


def build(force: bool = False) -> str:
    """Compile ``bitlinear_oracle.c`` into ``liboracle.so`` with gcc."""
    if force or not os.path.exists(_LIB_PATH) or \
            os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call([
            "gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
            "-fno-fast-math", "-Wall", "-Wextra", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        lib.oracle_abs_sum_exact.argtypes = [P, I64, P, ctypes.c_int]
        lib.oracle_abs_sum_exact.restype = ctypes.c_int
        lib.oracle_ternarize.argtypes = [P, I64, ctypes.c_float, ctypes.c_float, P]
        lib.oracle_ternarize.restype = None
        lib.oracle_pack_codes.argtypes = [P, I64, I64, P]
        lib.oracle_pack_codes.restype = I64
        lib.oracle_unpack_codes.argtypes = [P, I64, I64, P]
        lib.oracle_unpack_codes.restype = I64
        lib.oracle_act_quant.argtypes = [P, P, ctypes.c_double, I64, I64, P, P]
        lib.oracle_act_quant.restype = None
        lib.oracle_ternary_matmul.argtypes = [P, P, I64, I64, I64, P]
        lib.oracle_ternary_matmul.restype = None
        lib.oracle_ternary_matmul_at.argtypes = [P, P, I64, P, P, I64, P]
        lib.oracle_ternary_matmul_at.restype = None
        lib.oracle_dequant.argtypes = [P, P, P, I64, I64, P]
        lib.oracle_dequant.restype = None
        lib.oracle_act_quant_per_tensor.argtypes = [P, I64, I64, P, P]
        lib.oracle_act_quant_per_tensor.restype = None
        _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


# --------------------------------------------------------------------------
# rounding of an exact rational to binary32
# --------------------------------------------------------------------------

def rational_to_f32(num: int, den: int) -> np.float32:
    """num/den (num >= 0, den > 0) rounded once to binary32, nearest, ties to even.

    Subnormal results keep the 2^-149 quantum; results at or above 2^128 after
    rounding are +Inf.
    """
    if num < 0 or den <= 0:
        raise ValueError("need num >= 0 and den > 0")
    if num == 0:
        return np.float32(0.0)
    # e with 2^e <= num/den < 2^(e+1)
    e = num.bit_length() - den.bit_length()
    while (num << max(0, -e)) < (den << max(0, e)):
        e -= 1
    while (num << max(0, -(e + 1))) >= (den << max(0, e + 1)):
        e += 1
    qexp = max(e - 23, -149)             # weight of the last kept bit
    if qexp >= 0:
        n2, d2 = num, den << qexp
    else:
        n2, d2 = num << (-qexp), den
    q, r = divmod(n2, d2)
    if 2 * r > d2 or (2 * r == d2 and (q & 1)):
        q += 1
    if q.bit_length() + qexp > 128:
        return np.float32(np.inf)
    return np.float32(np.ldexp(float(q), qexp))


# --------------------------------------------------------------------------
# weights: absmean, ternarize, pack
# --------------------------------------------------------------------------

def abs_sum_units(w: np.ndarray) -> int:
    """Exact sum of |w| over a binary32 array, as an integer count of 2^-149."""
    lib = _load()
    w = np.ascontiguousarray(w, dtype=np.float32)
    digits = np.zeros(12, dtype=np.uint32)
    rc = lib.oracle_abs_sum_exact(_ptr(w), w.size, _ptr(digits), 12)
    if rc == -1:
        raise ValueError("non-finite weight")
    if rc != 0:
        raise RuntimeError(f"oracle_abs_sum_exact rc={rc}")
    return sum(int(d) << (32 * i) for i, d in enumerate(digits))


def absmean_gamma(w: np.ndarray) -> np.float32:
    """[P4-eq] item 1: gamma = (1/nm) sum |W_ij|, the exact mean rounded once to binary32."""
    if w.size == 0:
        raise ValueError("empty weight matrix")
    return rational_to_f32(abs_sum_units(w), w.size << 149)


def ternarize(w: np.ndarray, gamma: np.float32, eps: np.float32 = EPS_W) -> np.ndarray:
    """[P4-eq] item 1 / [P4-code] weight_quant: Clip(Round(W/(gamma+eps)), -1, 1), int8."""
    lib = _load()
    w = np.ascontiguousarray(w, dtype=np.float32)
    q = np.empty(w.shape, dtype=np.int8)
    lib.oracle_ternarize(_ptr(w), w.size, ctypes.c_float(gamma), ctypes.c_float(eps), _ptr(q))
    return q


def pack_codes(q: np.ndarray) -> np.ndarray:
    """[P5-lut] 2-bit codes, 4 per byte, 00=0 01=+1 10=-1; [N,K] int8 -> [N,K/4] uint8."""
    lib = _load()
    q = np.ascontiguousarray(q, dtype=np.int8)
    N, K = q.shape
    if K % 4:
        raise ValueError("K must be a multiple of 4")
    out = np.empty((N, K // 4), dtype=np.uint8)
    bad = lib.oracle_pack_codes(_ptr(q), N, K, _ptr(out))
    if bad:
        raise ValueError(f"{bad} values outside {{-1,0,1}}")
    return out


def unpack_codes(packed: np.ndarray, K: int, strict: bool = True) -> np.ndarray:
    """Inverse of :func:`pack_codes`; [N,K/4] uint8 -> [N,K] int8."""
    lib = _load()
    packed = np.ascontiguousarray(packed, dtype=np.uint8)
    N = packed.shape[0]
    if packed.shape[1] * 4 != K:
        raise ValueError("packed width must be K/4")
    q = np.empty((N, K), dtype=np.int8)
    bad = lib.oracle_unpack_codes(_ptr(packed), N, K, _ptr(q))
    if bad and strict:
        raise ValueError(f"{bad} invalid 11 codes")
    return q


def pack_weights_per_channel(w: np.ndarray, eps: np.float32 = EPS_W):
    """[P2-wr] per-output-channel scale s in R^N: the absmean of [P4-eq] item 1 taken
    over each output row, gamma_n = (1/K) sum_k |W_nk| (the exact mean rounded once to
    binary32), and W_q[n] = Clip(Round(W[n] / (gamma_n + eps)), -1, 1).  READING: the
    page gives the per-channel form but not how s is obtained; the row absmean is the
    plainest reading that keeps the page's ternarization.  The page stores s in FP16;
    here it stays binary32 like the per-tensor gamma.
    Returns (packed [N, K/4], gammas float32 [N], w_q int8 [N, K])."""
    w = np.ascontiguousarray(w, dtype=np.float32)
    gammas = np.array([absmean_gamma(row) for row in w], dtype=np.float32)
    q = np.stack([ternarize(row, g, eps) for row, g in zip(w, gammas)]) if len(w) else np.zeros(w.shape, np.int8)
    return pack_codes(q), gammas, q


def pack_weights(w: np.ndarray, eps: np.float32 = EPS_W):
    """absmean gamma, ternary codes and packed bytes of one latent matrix W [N,K] fp32."""
    gamma = absmean_gamma(w)
    q = ternarize(w, gamma, eps)
    return pack_codes(q), gamma, q


# --------------------------------------------------------------------------
# activations
# --------------------------------------------------------------------------

def act_quant(x_bits: np.ndarray, gain_bits: np.ndarray | None, rms_eps: float):
    """[P4-code] RMSNorm + activation_quant and [P4-eq] item 2, per token row.

    x_bits: [M,K] uint16 bf16 patterns; gain_bits: [K] uint16 or None;
    rms_eps < 0 disables RMSNorm.  Returns (x_q int8 [M,K], sigma float64 [M]).
    As activation_quant, the max of the normalized row is clamped at 1e-8: rows
    below it (zeros, tiny values) take 1e-8 as their max, and their codes are
    formed from x * r * g in binary32 (see bitlinear_oracle.c).
    """
    lib = _load()
    x_bits = np.ascontiguousarray(x_bits, dtype=np.uint16)
    M, K = x_bits.shape
    if gain_bits is not None:
        gain_bits = np.ascontiguousarray(gain_bits, dtype=np.uint16)
        assert gain_bits.shape == (K,)
    xq = np.empty((M, K), dtype=np.int8)
    sigma = np.empty(M, dtype=np.float64)
    lib.oracle_act_quant(_ptr(x_bits), _ptr(gain_bits) if gain_bits is not None else None,
                         float(rms_eps), M, K, _ptr(xq), _ptr(sigma))
    return xq, sigma


def act_quant_per_tensor(x_bits: np.ndarray):
    """[P5-aq] per-tensor absmax quantization with Q_b = 128 (no RMSNorm).

    x_bits: [M,K] uint16 bf16 patterns.  Returns (x_q int8 [M,K] in [-128, 127],
    sigma float64 [M], every entry max|x| / 128)."""
    lib = _load()
    x_bits = np.ascontiguousarray(x_bits, dtype=np.uint16)
    M, K = x_bits.shape
    xq = np.empty((M, K), dtype=np.int8)
    sigma = np.empty(M, dtype=np.float64)
    lib.oracle_act_quant_per_tensor(_ptr(x_bits), M, K, _ptr(xq), _ptr(sigma))
    return xq, sigma


# --------------------------------------------------------------------------
# contraction and dequantization
# --------------------------------------------------------------------------

def ternary_matmul(xq: np.ndarray, wq: np.ndarray) -> np.ndarray:
    """[P4-eq] item 3 / [P5-lut]: acc[t,n] = sum_k W_q[n,k] x_q[t,k] by add/skip/subtract, int32."""
    lib = _load()
    xq = np.ascontiguousarray(xq, dtype=np.int8)
    wq = np.ascontiguousarray(wq, dtype=np.int8)
    M, K = xq.shape
    N, K2 = wq.shape
    assert K == K2
    acc = np.empty((M, N), dtype=np.int32)
    lib.oracle_ternary_matmul(_ptr(xq), _ptr(wq), M, N, K, _ptr(acc))
    return acc


def ternary_matmul_at(xq: np.ndarray, wq: np.ndarray, ts: np.ndarray, ns: np.ndarray) -> np.ndarray:
    """:func:`ternary_matmul` at the listed (t, n) positions only."""
    lib = _load()
    xq = np.ascontiguousarray(xq, dtype=np.int8)
    wq = np.ascontiguousarray(wq, dtype=np.int8)
    ts = np.ascontiguousarray(ts, dtype=np.int64)
    ns = np.ascontiguousarray(ns, dtype=np.int64)
    assert ts.shape == ns.shape and xq.shape[1] == wq.shape[1]
    assert (ts < xq.shape[0]).all() and (ns < wq.shape[0]).all()
    acc = np.empty(ts.shape, dtype=np.int32)
    lib.oracle_ternary_matmul_at(_ptr(xq), _ptr(wq), xq.shape[1], _ptr(ts), _ptr(ns), ts.size, _ptr(acc))
    return acc


def dequant(acc: np.ndarray, sigma: np.ndarray, w_scale: np.ndarray) -> np.ndarray:
    """[P4-eq] item 4: y[t,n] = acc[t,n] * sigma[t] * w_scale[n] (gamma*max|n|/Q_b), float64."""
    lib = _load()
    acc = np.ascontiguousarray(acc, dtype=np.int32)
    sigma = np.ascontiguousarray(sigma, dtype=np.float64)
    w_scale = np.ascontiguousarray(w_scale, dtype=np.float64)
    M, N = acc.shape
    assert sigma.shape == (M,) and w_scale.shape == (N,)
    y = np.empty((M, N), dtype=np.float64)
    lib.oracle_dequant(_ptr(acc), _ptr(sigma), _ptr(w_scale), M, N, _ptr(y))
    return y


def bitlinear_forward(x_bits, gain_bits, rms_eps, w_latent, eps=EPS_W):
    """One BitLinear layer end to end ([P4-code] BitLinear.forward, integer form).

    Returns a dict with x_q, sigma, gamma, w_q, packed, acc and y (float64).
    """
    packed, gamma, wq = pack_weights(w_latent, eps)
    xq, sigma = act_quant(x_bits, gain_bits, rms_eps)
    acc = ternary_matmul(xq, wq)
    y = dequant(acc, sigma, np.full(wq.shape[0], float(gamma)))
    return dict(x_q=xq, sigma=sigma, gamma=gamma, w_q=wq, packed=packed, acc=acc, y=y)


# --------------------------------------------------------------------------
# the linear stack of a transformer layer
# --------------------------------------------------------------------------

def relu2_gate_bits(gate32: np.ndarray, up32: np.ndarray) -> np.ndarray:
    """h = bf16(fl32(fl32(max(gate, 0)^2) * up)) as bf16 bit patterns.

    The FFN gate of the 2B-parameter BitNet b1.58 models is squared ReLU; the
    block of [P5-block] uses SiLU in the same place.  gate32 and up32 are
    binary32 values (the BitLinear outputs); each product is one binary32
    rounding, then one rounding to bf16 (nearest even).
    """
    g = np.ascontiguousarray(gate32, dtype=np.float32)
    u = np.ascontiguousarray(up32, dtype=np.float32)
    r = np.maximum(g, np.float32(0.0))
    h = np.multiply(np.multiply(r, r, dtype=np.float32), u, dtype=np.float32)
    return f32_to_bf16_bits(h)


def bitlinear_f32(x_bits, gain_bits, rms_eps, wq, w_scale):
    """One BitLinear with its RMSNorm ([P4-code] BitLinear.forward): the fp64
    output of :func:`dequant` rounded once to binary32."""
    xq, sigma = act_quant(x_bits, gain_bits, rms_eps)
    return dequant(ternary_matmul(xq, wq), sigma, w_scale).astype(np.float32)


def block_layer(x_bits, layer: dict, rms_eps: float):
    """One layer of the linear stack on the bf16 residual stream x [M, H].

    Follows the block of [P5-block] with every projection a BitLinear (its
    RMSNorm standing in for the block's LayerNorms):
        q = bf16(BitLinear_qkv(x))[:, :H]    -- READING: attention is not part
                                                of this stack, the query slice
                                                stands in for its output
        x = bf16(fl32(x + BitLinear_o(q)))
        g | u = BitLinear_gate_up(x)         (fp32, gate rows then up rows)
        h = relu2_gate_bits(g, u)
        x = bf16(fl32(x + BitLinear_down(h)))
    ``layer`` holds int8 ternary matrices ``qkv``, ``o``, ``gate_up``, ``down``,
    per-row float scales ``*_scale`` and bf16 gains ``gain_*`` (bit patterns).
    Returns the new x as bf16 bits.
    """
    x_bits = np.ascontiguousarray(x_bits, dtype=np.uint16)
    H = x_bits.shape[1]
    F = layer["down"].shape[1]
    x32 = bf16_bits_to_f64(x_bits).astype(np.float32)
    qkv = bitlinear_f32(x_bits, layer["gain_qkv"], rms_eps, layer["qkv"], layer["qkv_scale"])
    q_bits = f32_to_bf16_bits(np.ascontiguousarray(qkv[:, :H]))
    o = bitlinear_f32(q_bits, layer["gain_o"], rms_eps, layer["o"], layer["o_scale"])
    x_bits = f32_to_bf16_bits(np.add(x32, o, dtype=np.float32))
    x32 = bf16_bits_to_f64(x_bits).astype(np.float32)
    gu = bitlinear_f32(x_bits, layer["gain_gate_up"], rms_eps, layer["gate_up"], layer["gate_up_scale"])
    h_bits = relu2_gate_bits(gu[:, :F], gu[:, F:])
    d = bitlinear_f32(h_bits, layer["gain_down"], rms_eps, layer["down"], layer["down_scale"])
    return f32_to_bf16_bits(np.add(x32, d, dtype=np.float32))


# --------------------------------------------------------------------------
# helpers shared by the tests (no arithmetic of the method)
# --------------------------------------------------------------------------

def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """binary32 -> bf16 bit patterns, round to nearest even (finite inputs)."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def bf16_bits_to_f64(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def exact_fraction_f32(v) -> Fraction:
    return Fraction(float(np.float32(v)))
