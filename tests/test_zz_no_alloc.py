"""The allocation-free weight packer against the regular one.

bitlinear_pack_weights_static exists for callers that cannot allocate device
memory (a plugin handed only pre-sized buffers, or a latency-critical path where
cudaMalloc could synchronize the device); it keeps its scratch in a fixed array
inside the library.  This test calls it through the C ABI twice in a row, on two
different matrices, and requires exactly the packed bytes, per-row scales and
gamma that bitlinear_pack_weights (with a caller workspace) produces -- the
second call also shows that what the first call left in the shared array does
not leak into the next result.
"""
import ctypes

import numpy as np
import pytest
import torch

import bitlinear_rmsnorm_token_int8_b300 as bl
from bitlinear_rmsnorm_token_int8_b300 import synth

pytestmark = pytest.mark.gpu


def _static_pack(L, W):
    N, K = W.shape
    packed = torch.empty(bl.bitlinear_packed_bytes(N, K), dtype=torch.uint8, device=W.device)
    w_scale = torch.empty(N, dtype=torch.float32, device=W.device)
    gamma = torch.empty(4, dtype=torch.float32, device=W.device)
    fn = L.bitlinear_pack_weights_static
    fn.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_float, ctypes.c_void_p,
                   ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    fn.restype = ctypes.c_int
    st = fn(W.data_ptr(), N, K, 1e-5, packed.data_ptr(), w_scale.data_ptr(), gamma.data_ptr(),
            torch.cuda.current_stream().cuda_stream)
    assert st == 0, bl.STATUS.get(st, st)
    return packed, w_scale, gamma[:1]


def test_static_scratch_packer_matches_workspace_packer_on_two_calls():
    assert torch.cuda.is_available()
    L = bl.lib()
    shapes = [(2560, 2560), (37, 6912)]          # second call: different size and gamma
    for i, (N, K) in enumerate(shapes):
        W = synth.latent_weights(N, K, seed=77 + i).cuda()
        if i == 1:
            W = W * 3.0                            # a different absmean than the first call
        p_ref, s_ref, g_ref = bl.bitlinear_pack_weights(W)
        p_st, s_st, g_st = _static_pack(L, W)
        torch.cuda.synchronize()
        assert torch.equal(p_st, p_ref)
        assert torch.equal(s_st, s_ref)
        assert torch.equal(g_st, g_ref)
    assert bl.bitlinear_get_device_error() == 0


def test_static_scratch_packer_rejects_sizes_beyond_its_limit():
    L = bl.lib()
    fn = L.bitlinear_pack_weights_static
    fn.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_float, ctypes.c_void_p,
                   ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    fn.restype = ctypes.c_int
    fake = 1 << 20
    assert fn(fake, 1 << 20, 1 << 12, 1e-5, fake, fake, None, None) == 2   # N*K >= 2^32
