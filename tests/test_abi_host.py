"""Host-side checks of the C ABI that need no GPU: the library loads, exports
every function that include/bitlinear.h declares, sizes its buffers, and
rejects bad arguments before touching the device."""
import ctypes
import os
import re

import pytest

import bitlinear_rmsnorm_token_int8_b300 as bl
from bitlinear_rmsnorm_token_int8_b300 import build as blbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER_DIR = os.path.join(ROOT, "include")

OK, ERR_NULL, ERR_SHAPE, ERR_ALIGN, ERR_DTYPE, ERR_DEVICE, ERR_CUDA, ERR_TIMEOUT, ERR_WS, ERR_NF = range(10)
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


def test_status_strings_and_version(L):
    assert L.bitlinear_abi_version() == 1
    for s in range(10):
        assert L.bitlinear_status_string(s)
    assert L.bitlinear_status_string(99) == b"unknown status"


def test_sizes(L):
    assert L.bitlinear_packed_bytes(4096, 14336) == 4096 * 14336 // 4
    assert L.bitlinear_packed_bytes(-1, 4) == 0
    assert L.bitlinear_pack_workspace_bytes(1, 4) >= 2048
    for M, N, K in [(1, 2560, 2560), (16, 28672, 4096), (2048, 14336, 4096)]:
        assert L.bitlinear_forward_workspace_bytes(M, N, K) >= 0


def _fwd(L, x=FAKE, s=FAKE, p=FAKE, w=FAKE, M=4, N=512, K=256, dt=0, y=FAKE, acc=None, ws=FAKE,
         wsb=1 << 30):
    return L.bitlinear_forward(x, s, p, w, M, N, K, dt, y, acc, ws, wsb, None)


def test_forward_argument_errors(L):
    assert _fwd(L, x=None) == ERR_NULL
    assert _fwd(L, y=None) == ERR_NULL
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
    # valid arguments: only now is the device consulted (none here, or not sm_103)
    import torch
    if not torch.cuda.is_available():
        assert _fwd(L) == ERR_DEVICE


def test_quant_act_argument_errors(L):
    q = L.bitlinear_quant_act
    assert q(None, None, 1e-5, 4, 256, FAKE, FAKE, None) == ERR_NULL
    assert q(None, None, 1e-5, 0, 256, None, None, None) == OK
    assert q(FAKE, None, 1e-5, 4, 12, FAKE, FAKE, None) == ERR_SHAPE
    assert q(FAKE, None, 1e-5, 4, 65536 + 8, FAKE, FAKE, None) == ERR_SHAPE
    assert q(FAKE, None, 1e-5, -2, 256, FAKE, FAKE, None) == ERR_SHAPE
    assert q(FAKE, FAKE + 2, 1e-5, 4, 256, FAKE, FAKE, None) == ERR_ALIGN
    import torch
    if not torch.cuda.is_available():
        assert q(FAKE, None, 1e-5, 4, 256, FAKE, FAKE, None) == ERR_DEVICE


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
