"""GPU parity of the scale-granularity variants against the CPU oracle:

* bitlinear_pack_weights_per_channel (page "BitNet-2B-4T", Weight
  Representation: a scale per output channel): gamma_n and the codes bit-exact;
* bitlinear_quant_act_per_tensor (page "BitNet 1-bit LLM Inference Framework",
  BitLinear.activation_quantize: one scale for the tensor, Q_b = 128, codes in
  [-128, 127]): codes bit-exact, the scale exact (gamma / 2^7);
* bitlinear_forward on their outputs, on every route: int32 accumulators
  bit-exact, fp32 outputs within 1e-6 relative (as the main path's parity).
"""
import json
import os

import numpy as np
import pytest
import torch

import bitlinear_rmsnorm_token_int8_b300 as bl
import oracle
from bitlinear_rmsnorm_token_int8_b300 import layout, synth

pytestmark = pytest.mark.gpu

F32_RTOL = 1e-6
GOLDEN = json.load(open(os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "worked_examples.json")))


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    bl.lib()
    yield
    assert bl.bitlinear_get_device_error() == 0


def bits_tensor(a32: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(oracle.f32_to_bf16_bits(a32).view(np.int16)).view(torch.bfloat16)


def gpu_pack_pc(W: np.ndarray):
    N, K = W.shape
    packed, ws = bl.bitlinear_pack_weights_per_channel(torch.from_numpy(W).cuda())
    torch.cuda.synchronize()
    return layout.canonical_from_tiled(packed.cpu().numpy(), N, K), ws.cpu().numpy(), packed, ws


@pytest.mark.parametrize("N,K", [(2, 4), (16, 512), (37, 2560), (130, 1028), (300, 6912)])
def test_pack_per_channel_matches_oracle(N, K):
    rng = np.random.default_rng(N + K)
    if (N, K) == (2, 4):
        W = np.array(GOLDEN["weights_per_channel_2x4"]["W"], dtype=np.float32)
    else:
        # rows of very different magnitudes, so one scale per row matters
        W = (rng.standard_normal((N, K)) * 0.02 * np.exp2(rng.integers(-8, 8, (N, 1)))).astype(np.float32)
        W[0, :3] = [1e-40, -3e-39, 3e38]          # subnormals and a huge value in one row
    canon, ws, _, _ = gpu_pack_pc(W)
    o_packed, o_g, o_wq = oracle.pack_weights_per_channel(W)
    assert (ws == o_g).all()
    assert (canon == o_packed).all()


def test_forward_with_per_channel_scales_matches_oracle():
    rng = np.random.default_rng(3)
    M, N, K = 5, 400, 2560
    W = (rng.standard_normal((N, K)) * 0.02 * np.exp2(rng.integers(-4, 4, (N, 1)))).astype(np.float32)
    _, ws_np, packed, ws = gpu_pack_pc(W)
    x = synth.activations(M, K, seed=9)
    xq, sc = bl.bitlinear_quant_act(x.cuda(), None, 1e-5)
    acc = torch.empty((M, N), dtype=torch.int32, device="cuda")
    y = bl.bitlinear_forward(xq, sc, packed, ws, out_dtype=torch.float32, acc_debug=acc)
    torch.cuda.synchronize()
    o_xq, o_sig = oracle.act_quant(synth.bf16_bits(x), None, float(np.float32(1e-5)))
    _, o_g, o_wq = oracle.pack_weights_per_channel(W)
    o_acc = oracle.ternary_matmul(o_xq, o_wq)
    assert (acc.cpu().numpy() == o_acc).all()
    o_y = oracle.dequant(o_acc, o_sig, o_g.astype(np.float64))
    yv = y.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(yv - o_y) <= F32_RTOL * np.abs(o_y))


@pytest.mark.parametrize("key", ["act_per_tensor_q128", "act_per_tensor_tiny"])
def test_quant_per_tensor_golden(key):
    ex = GOLDEN[key]
    x = np.array(ex["x"], dtype=np.float32)
    M, K = x.shape
    xp = np.zeros((M, 8), dtype=np.float32)                 # K padded to 8 with zeros (no effect on max or codes)
    xp[:, :K] = x
    xq, sc = bl.bitlinear_quant_act_per_tensor(bits_tensor(xp).cuda())
    torch.cuda.synchronize()
    assert xq.cpu().numpy()[:, :K].tolist() == ex["x_q"]
    want = ex["sigma"] if "sigma" in ex else 2.0 ** ex["sigma_log2"]
    assert (sc.cpu().numpy() == np.float32(want)).all()


@pytest.mark.parametrize("M,K", [(1, 8), (4, 256), (16, 4096), (33, 2560), (600, 4104), (3, 65536)])
def test_quant_per_tensor_matches_oracle(M, K):
    x = synth.activations(M, K, seed=M * 7 + K, outliers=True)
    xq, sc = bl.bitlinear_quant_act_per_tensor(x.cuda())
    torch.cuda.synchronize()
    oq, osig = oracle.act_quant_per_tensor(synth.bf16_bits(x))
    assert (xq.cpu().numpy() == oq).all()
    assert (sc.cpu().numpy().astype(np.float64) == osig).all()     # gamma / 128 is exact


@pytest.mark.parametrize("M,N,K", [(1, 2560, 2560), (2, 3840, 2560), (8, 1040, 4096), (64, 512, 1536),
                                   (300, 400, 6912)])
def test_forward_on_per_tensor_codes_every_route(M, N, K):
    # the per-tensor codes reach -128 (the clip is asymmetric); every contraction route
    # (int8 codes on the CUDA cores, the operand form on tcgen05 decode and prefill)
    x = synth.activations(M, K, seed=M + N, outliers=True)
    W = synth.latent_weights(N, K, seed=N + 1)
    packed, w_scale, gamma = bl.bitlinear_pack_weights(W.cuda())
    xq, sc, ops = bl.bitlinear_quant_act_per_tensor(x.cuda(), x_ops=True)
    accs = []
    for use_ops in (False, True):
        acc = torch.empty((M, N), dtype=torch.int32, device="cuda")
        y = bl.bitlinear_forward(None if use_ops else xq, sc, packed, w_scale, out_dtype=torch.float32,
                                 acc_debug=acc, x_ops=ops if use_ops else None, K=K)
        torch.cuda.synchronize()
        accs.append((acc.cpu(), y.cpu()))
    assert torch.equal(accs[0][0], accs[1][0]) and torch.equal(accs[0][1], accs[1][1])
    oq, osig = oracle.act_quant_per_tensor(synth.bf16_bits(x))
    _, o_g, o_wq = oracle.pack_weights(W.numpy())
    o_acc = oracle.ternary_matmul(oq, o_wq)
    assert (accs[0][0].numpy() == o_acc).all()
    o_y = oracle.dequant(o_acc, osig, np.full(N, float(o_g)))
    yv = accs[0][1].numpy().astype(np.float64)
    assert np.all(np.abs(yv - o_y) <= F32_RTOL * np.abs(o_y))


@pytest.mark.parametrize("M,K", [(1, 65536), (8, 65536), (40, 14336)])
def test_all_minus_128_codes_at_the_longest_rows(M, K):
    # a constant negative tensor quantizes to -128 everywhere; against all-(+1) weights
    # every accumulator is -128 K (-2^23 at K = 65536), exact on every route
    x = torch.full((M, K), -0.75, dtype=torch.bfloat16)
    xq, sc, ops = bl.bitlinear_quant_act_per_tensor(x.cuda(), x_ops=True)
    assert (xq == -128).all()
    N = 128
    W = torch.full((N, K), 0.02)
    packed, w_scale, _ = bl.bitlinear_pack_weights(W.cuda())
    for use_ops in (False, True):
        acc = torch.empty((M, N), dtype=torch.int32, device="cuda")
        bl.bitlinear_forward(None if use_ops else xq, sc, packed, w_scale, out_dtype=torch.float32, acc_debug=acc,
                             x_ops=ops if use_ops else None, K=K)
        torch.cuda.synchronize()
        assert (acc.cpu() == -128 * K).all()
