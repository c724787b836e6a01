"""Host-side checks of the C ABI that need no GPU: the library loads, exports
every function that include/bitlinear.h declares, sizes its buffers, and
rejects bad arguments before touching the device."""
import ctypes

import numpy as np
import os
import re

import pytest

import bitlinear_rmsnorm_token_int8_b300 as bl
from bitlinear_rmsnorm_token_int8_b300 import build as blbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER_DIR = os.path.join(ROOT, "include")

(OK, ERR_NULL, ERR_SHAPE, ERR_ALIGN, ERR_DTYPE, ERR_DEVICE, ERR_CUDA, ERR_TIMEOUT, ERR_WS, ERR_NF,
 ERR_FLAGS) = range(11)
FAKE = 1 << 20        # an aligned, never-dereferenced address


@pytest.fixture(scope="module")
def L():
    blbuild.build()
    return bl.lib()


def declared_functions():
    names = set()
    for fn in os.listdir(HEADER_DIR):
        if fn.endswith(".h"):
            text = open(os.path.join(HEADER_DIR, fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names.update(re.findall(r"\b(bitlinear_\w+)\s*\(", text))
    return sorted(names)


def test_library_exports_every_declared_function(L):
    names = declared_functions()
    assert "bitlinear_forward" in names and "bitlinear_quant_act" in names
    for n in names:
        assert hasattr(L, n), f"{n} declared in include/ but not exported"


def test_codes_route_limit_matches_the_header():
    text = open(os.path.join(HEADER_DIR, "bitlinear.h")).read()
    m = re.search(r"#define BITLINEAR_CODES_MAX_M (\d+)", text)
    assert m and int(m.group(1)) == bl.CODES_MAX_M


def test_codes_route_needs_no_workspace(L):
    # bitlinear_forward given x_q: no scratch where the int8-code kernel takes it
    ws = L.bitlinear_forward_workspace_bytes
    assert ws(1, 2560, 2560) == 0 and ws(1, 4096, 65536) == 0 and ws(2, 3840, 2560) == 0
    assert ws(2, 28672, 4096) == 0 and ws(2, 4096, 37376) == 0
    assert ws(2, 4096, 65536) == L.bitlinear_act_ops_bytes(2, 65536)   # two tokens' codes do not fit
    assert ws(3, 2560, 2560) == L.bitlinear_act_ops_bytes(3, 2560)     # three tokens: tcgen05
    assert ws(64, 2560, 2560) == L.bitlinear_act_ops_bytes(64, 2560)


def test_linear_route(L):
    route = L.bitlinear_linear_route
    assert route(1, 2560, 2560) == bl.ROUTE_FUSED            # one token, K <= 8192: one kernel
    assert route(1, 4096, 8192) == bl.ROUTE_FUSED
    assert route(1, 4096, 14336) == bl.ROUTE_FUSED           # up to 16384 on the persistent kernel
    assert route(1, 512, 14336) == bl.ROUTE_CODES            # a small matrix: quant + small-CTA codes kernel
    assert route(1, 4096, 16896) == bl.ROUTE_CODES           # longer K: quant + codes kernel
    assert route(2, 3840, 2560) == bl.ROUTE_CODES            # two tokens: quant + codes kernel
    assert route(2, 28672, 4096) == bl.ROUTE_CODES
    assert route(2, 4096, 14336) == bl.ROUTE_CODES
    assert route(2, 4096, 65536) == bl.ROUTE_DECODE          # two tokens' codes do not fit: tcgen05
    assert route(3, 2560, 2560) == bl.ROUTE_DECODE
    assert route(4, 28672, 4096) == bl.ROUTE_DECODE
    assert route(32, 2560, 2560) == bl.ROUTE_DECODE
    assert route(33, 2560, 2560) == bl.ROUTE_PREFILL
    assert route(0, 2560, 2560) == -1 and route(1, 24, 2560) == -1 and route(1, 2560, 100) == -1
    for name, value in [("FUSED", 0), ("CODES", 1), ("DECODE", 2), ("PREFILL", 3)]:
        assert re.search(rf"#define BITLINEAR_ROUTE_{name} {value}\b", open(os.path.join(HEADER_DIR, "bitlinear.h")).read())
        assert getattr(bl, f"ROUTE_{name}") == value


def test_status_strings_and_version(L):
    assert L.bitlinear_abi_version() == 2
    for s in range(11):
        assert L.bitlinear_status_string(s)
    assert L.bitlinear_status_string(99) == b"unknown status"


def test_prefill_cluster_size_needs_local_device_memory(L):
    # the cluster-of-2 prefill kernel multicasts activation blocks; it is chosen only for
    # operands in the current device's own memory, never for a host address
    host = np.zeros(1 << 16, dtype=np.uint8)
    addr = host.ctypes.data
    assert L.bitlinear_prefill_cluster_size(addr, 2048, 14336, 4096) == 1
    assert L.bitlinear_prefill_cluster_size(addr, 2048, 128, 4096) == 1
    assert L.bitlinear_prefill_cluster_size(addr, 8, 14336, 4096) == -1      # decode route
    assert L.bitlinear_prefill_cluster_size(None, 2048, 14336, 4096) == -1
    assert L.bitlinear_prefill_cluster_size(addr, 2048, 100, 4096) == -1     # rejected shape


def test_sizes(L):
    assert L.bitlinear_packed_bytes(4096, 14336) == 4096 * 14336 // 4
    assert L.bitlinear_packed_bytes(-1, 4) == 0
    assert L.bitlinear_pack_workspace_bytes(1, 4) >= 2048
    for M, N, K in [(1, 2560, 2560), (16, 28672, 4096), (2048, 14336, 4096)]:
        assert L.bitlinear_forward_workspace_bytes(M, N, K) >= 0
    # operand form: two e4m3 planes, K padded to a multiple of 512
    assert L.bitlinear_act_ops_bytes(8, 2560) == 2 * 8 * 2560
    assert L.bitlinear_act_ops_bytes(3, 384) == 2 * 8 * 512        # decode layout: tokens padded to 8
    assert L.bitlinear_act_ops_bytes(17, 1024) == 2 * 24 * 1024
    assert L.bitlinear_act_ops_bytes(32, 640) == 2 * 32 * 1024
    assert L.bitlinear_act_ops_bytes(-1, 384) == 0
    assert L.bitlinear_act_ops_bytes(33, 384) == 2 * 256 * 512      # prefill layout: tokens padded to 256


def _fwd(L, x=FAKE, s=FAKE, ops=None, p=FAKE, w=FAKE, M=4, N=512, K=256, dt=0, y=FAKE, acc=None,
         ws=FAKE, wsb=1 << 30, flags=0, pf=None, pfb=0):
    return L.bitlinear_forward(x, s, ops, p, w, M, N, K, dt, y, acc, ws, wsb, pf, pfb, flags, None)


def test_forward_argument_errors(L):
    assert _fwd(L, x=None) == ERR_NULL
    assert _fwd(L, y=None) == ERR_NULL
    assert _fwd(L, flags=2) == ERR_FLAGS
    # more than CODES_MAX_M tokens and no x_ops: x_q is converted in the workspace
    assert _fwd(L, M=16, ws=None) == ERR_WS
    assert _fwd(L, M=16, wsb=L.bitlinear_forward_workspace_bytes(16, 512, 256) - 1) == ERR_WS
    assert _fwd(L, ops=FAKE + 8) == ERR_ALIGN
    assert _fwd(L, M=0, x=None, y=None, s=None) == OK       # empty: nothing to touch
    assert _fwd(L, K=100) == ERR_SHAPE
    assert _fwd(L, K=0) == ERR_SHAPE
    assert _fwd(L, N=8) == ERR_SHAPE
    assert _fwd(L, N=520) == ERR_SHAPE
    assert _fwd(L, M=-1) == ERR_SHAPE
    assert _fwd(L, K=65536 + 128) == ERR_SHAPE
    assert _fwd(L, dt=7) == ERR_DTYPE
    assert _fwd(L, x=FAKE + 4) == ERR_ALIGN
    assert _fwd(L, acc=FAKE + 8) == ERR_ALIGN
    assert _fwd(L, pf=FAKE + 8, pfb=4096) == ERR_ALIGN      # the L2 prefetch range must be 16-byte aligned
    # valid arguments: only now is the device consulted (none here, or not sm_103)
    import torch
    if not torch.cuda.is_available():
        assert _fwd(L) == ERR_DEVICE
        assert _fwd(L, x=None, ops=FAKE, ws=None, flags=1) == ERR_DEVICE   # x_ops alone suffices
        assert _fwd(L, M=2, ws=None) == ERR_DEVICE            # one or two tokens: x_q alone suffices
        assert _fwd(L, pf=FAKE, pfb=100) == ERR_DEVICE        # any size: rounded down to 16 bytes


def test_quant_act_argument_errors(L):
    def q(x, g, eps, M, K, xq, sc, ops=None, flags=0):
        return L.bitlinear_quant_act(x, g, eps, M, K, xq, sc, ops, flags, None)
    assert q(None, None, 1e-5, 4, 256, FAKE, FAKE) == ERR_NULL
    assert q(None, None, 1e-5, 0, 256, None, None) == OK
    assert q(FAKE, None, 1e-5, 4, 12, FAKE, FAKE) == ERR_SHAPE
    assert q(FAKE, None, 1e-5, 4, 65536 + 8, FAKE, FAKE) == ERR_SHAPE
    assert q(FAKE, None, 1e-5, -2, 256, FAKE, FAKE) == ERR_SHAPE
    assert q(FAKE, FAKE + 2, 1e-5, 4, 256, FAKE, FAKE) == ERR_ALIGN
    assert q(FAKE, None, 1e-5, 4, 256, FAKE, FAKE, ops=FAKE + 4) == ERR_ALIGN
    assert q(FAKE, None, 1e-5, 4, 256, FAKE, FAKE, flags=4) == ERR_FLAGS
    import torch
    if not torch.cuda.is_available():
        assert q(FAKE, None, 1e-5, 4, 256, FAKE, FAKE) == ERR_DEVICE
        assert q(FAKE, None, 1e-5, 4, 256, FAKE, FAKE, ops=FAKE, flags=1) == ERR_DEVICE


def test_linear_forward_argument_errors(L):
    def lf(x=FAKE, g=None, p=FAKE, w=FAKE, M=4, N=512, K=256, dt=1, y=FAKE, xq=None, sc=None, acc=None,
           ws=None, wsb=0, flags=0, pf=None, pfb=0):
        return L.bitlinear_linear_forward(x, g, 1e-5, p, w, M, N, K, dt, y, xq, sc, acc, ws, wsb, pf, pfb, flags,
                                          None)
    assert lf(x=None) == ERR_NULL
    assert lf(p=None) == ERR_NULL
    assert lf(M=0, x=None, p=None, w=None, y=None) == OK
    assert lf(K=200) == ERR_SHAPE                   # the contraction needs K % 128 == 0
    assert lf(N=24) == ERR_SHAPE
    assert lf(M=-1) == ERR_SHAPE
    assert lf(dt=5) == ERR_DTYPE
    assert lf(flags=8) == ERR_FLAGS
    assert lf(g=FAKE + 2) == ERR_ALIGN
    assert lf(xq=FAKE + 8) == ERR_ALIGN
    assert lf(pf=FAKE + 4, pfb=64) == ERR_ALIGN
    # quantization into the workspace (operand form + scales), then the contraction
    assert L.bitlinear_linear_workspace_bytes(1, 2560, 2560) >= L.bitlinear_act_ops_bytes(1, 2560) + 4
    need = L.bitlinear_linear_workspace_bytes(64, 512, 256)
    assert need >= L.bitlinear_act_ops_bytes(64, 256) + 4 * 64
    assert lf(M=64) == ERR_WS
    assert lf(M=64, ws=FAKE, wsb=need - 1) == ERR_WS
    assert lf(M=64, ws=FAKE + 4, wsb=need) == ERR_ALIGN
    assert lf() == ERR_WS
    import torch
    if not torch.cuda.is_available():
        assert lf(M=64, ws=FAKE, wsb=need) == ERR_DEVICE


def test_pack_argument_errors(L):
    p = L.bitlinear_pack_weights
    ws = L.bitlinear_pack_workspace_bytes(8, 8)
    assert p(None, 8, 8, 1e-5, FAKE, FAKE, None, FAKE, ws, None) == ERR_NULL
    assert p(FAKE, 8, 6, 1e-5, FAKE, FAKE, None, FAKE, ws, None) == ERR_SHAPE
    assert p(FAKE, 0, 8, 1e-5, FAKE, FAKE, None, FAKE, ws, None) == ERR_SHAPE
    assert p(FAKE, 1 << 20, 1 << 12, 1e-5, FAKE, FAKE, None, FAKE, ws, None) == ERR_SHAPE
    assert p(FAKE, 8, 8, -1.0, FAKE, FAKE, None, FAKE, ws, None) == ERR_SHAPE
    assert p(FAKE, 8, 8, 1e-5, FAKE, FAKE, None, None, ws, None) == ERR_WS
    assert p(FAKE, 8, 8, 1e-5, FAKE, FAKE, None, FAKE, ws - 1, None) == ERR_WS
    assert p(FAKE, 8, 8, 1e-5, FAKE + 1, FAKE, None, FAKE, ws, None) == ERR_ALIGN
    import torch
    if not torch.cuda.is_available():
        assert p(FAKE, 8, 8, 1e-5, FAKE, FAKE, None, FAKE, ws, None) == ERR_DEVICE


def test_python_binding_rejects_cpu_tensors():
    import torch
    with pytest.raises(ValueError):
        bl.bitlinear_quant_act(torch.zeros(2, 16, dtype=torch.bfloat16))


def test_packed_layout_index_is_a_bijection_onto_the_data_bytes():
    from bitlinear_rmsnorm_token_int8_b300 import layout
    rng = np.random.default_rng(0)
    for N, K in [(1, 4), (16, 512), (37, 2560), (48, 6912), (3, 516)]:
        idx = layout.packed_index(N, K)
        assert idx.shape == (N, K // 4)
        assert len(np.unique(idx)) == idx.size and idx.min() >= 0 and idx.max() < layout.packed_bytes(N, K)
        canon = rng.integers(0, 256, (N, K // 4), dtype=np.uint8)
        tiled = layout.tiled_from_canonical(canon, K)
        assert (layout.canonical_from_tiled(tiled, N, K) == canon).all()
        # padding stays zero; the size matches the C ABI's
        assert tiled.sum() == canon.astype(np.int64).sum()
        assert layout.packed_bytes(N, K) == _lib_bytes(N, K)


def test_packed_layout_swizzle_example():
    # row 9 (tile 0, r = 9, r % 8 = 1), canonical byte 20 (segment 0, chunk 1, offset 4):
    # chunk 1 ^ 1 = 0 -> offset 9*128 + 0*16 + 4
    from bitlinear_rmsnorm_token_int8_b300 import layout
    assert layout.packed_index(16, 512)[9, 20] == 9 * 128 + 4
    # segment 1 of a full tile starts after the 128 rows of segment 0
    assert layout.packed_index(130, 1024)[0, 128] == 128 * 128
    # row 128 starts tile 1 after both segments of tile 0 (K = 1024 -> 2 segments)
    assert layout.packed_index(130, 1024)[128, 0] == 2 * 128 * 128
    # the last tile holds the 16 rows of N = 130 padded to 144: its segment blocks are 16 x 128 bytes
    assert layout.packed_index(130, 1024)[129, 128] == 2 * 128 * 128 + 16 * 128 + 1 * 128 + (0 ^ 1) * 16
    assert layout.packed_bytes(130, 1024) == 144 * 2 * 128


def _lib_bytes(N, K):
    blbuild.build()
    return bl.lib().bitlinear_packed_bytes(N, K)


def test_scale_variant_argument_errors(L):
    pc = L.bitlinear_pack_weights_per_channel
    assert pc(None, 8, 8, 1e-5, FAKE, FAKE, None) == ERR_NULL
    assert pc(FAKE, 8, 6, 1e-5, FAKE, FAKE, None) == ERR_SHAPE
    assert pc(FAKE, 8, 8, -1.0, FAKE, FAKE, None) == ERR_SHAPE
    assert pc(FAKE, 1 << 20, 1 << 12, 1e-5, FAKE, FAKE, None) == ERR_SHAPE
    assert pc(FAKE, 8, 8, 1e-5, FAKE + 4, FAKE, None) == ERR_ALIGN
    need = L.bitlinear_quant_act_per_tensor_workspace_bytes(100)
    assert need >= 400 and need % 256 == 0
    qt = L.bitlinear_quant_act_per_tensor
    assert qt(None, 4, 256, FAKE, FAKE, None, FAKE, need, 0, None) == ERR_NULL
    assert qt(FAKE, 4, 256, None, FAKE, None, FAKE, need, 0, None) == ERR_NULL
    assert qt(FAKE, 4, 12, FAKE, FAKE, None, FAKE, need, 0, None) == ERR_SHAPE
    assert qt(FAKE, 0, 256, None, None, None, None, 0, 0, None) == OK       # empty: nothing to touch
    assert qt(FAKE, 4, 256, FAKE, FAKE, None, None, 0, 0, None) == ERR_WS
    assert qt(FAKE, 4, 256, FAKE, FAKE, FAKE + 8, FAKE, need, 0, None) == ERR_ALIGN
    assert qt(FAKE, 4, 256, FAKE, FAKE, None, FAKE, need, 2, None) == ERR_FLAGS
    import torch
    if not torch.cuda.is_available():
        assert pc(FAKE, 8, 8, 1e-5, FAKE, FAKE, None) == ERR_DEVICE
        assert qt(FAKE, 4, 256, FAKE, FAKE, None, FAKE, need, 1, None) == ERR_DEVICE
