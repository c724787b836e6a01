"""GPU parity of bitlinear_block_forward (the BitLinear stack of transformer
layers) at the 2B-class layer dims (hidden 2560, QKV 3840, FFN 6912), two
layers, M = 1, 8 and 512 tokens, checked BitLinear by BitLinear on its exact
input (teacher forced): the block's trace gives every BitLinear's input as the
GPU formed it, the oracle quantizes and contracts that input, and

* int8 codes are bit-exact and token scales within 5e-7 relative;
* bf16 qkv is within 1 bf16 ulp of the oracle's fp64 output;
* fp32 gate|up is within 1e-6 relative;
* a residual sum x + y (bf16) is within half a bf16 ulp of the exact sum
  x + y_exact plus the fp32 error bound of y (3.9e-7 |y|, from sigma's 3.5
  fp32 ulp and the two roundings of the dequantization): the GPU rounds
  fl32(x + y_gpu) to bf16, so |gpu - exact| <= 2^-8 |exact| + 2^-24 |x + y| +
  3.9e-7 |y|.
Layer 1 is fed the GPU's own layer-0 output, so a rounding difference in an
intermediate never carries into the next check.  For M = 512 the contractions
are checked on 24 sampled tokens (all tokens' codes are checked).
"""
import numpy as np
import pytest
import torch

import bitlinear_rmsnorm_token_int8_b300 as bl
import oracle
from bitlinear_rmsnorm_token_int8_b300 import synth

pytestmark = pytest.mark.gpu

RMS_EPS = float(np.float32(1e-5))
SIGMA_RTOL = 5e-7
F32_RTOL = 1e-6
Y_RTOL = 3.9e-7
H, NQKV, F = 2560, 3840, 6912


def ulp_distance(a_bits, b_bits):
    def ordered(u):
        u = u.astype(np.int32)
        return np.where(u & 0x8000, -(u & 0x7FFF), u & 0x7FFF)
    return np.abs(ordered(a_bits) - ordered(b_bits))


def bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def make_layer(H, NQKV, F, seed):
    """Latent weights packed on the GPU; the oracle's copy from the oracle's own packer."""
    mats = {"qkv": [(NQKV, H)], "o": [(H, H)], "gate_up": [(F, H), (F, H)], "down": [(H, F)]}
    g_layer, o_layer = {}, {}
    for j, (name, shapes) in enumerate(mats.items()):
        Ws = [synth.latent_weights(n, k, seed=seed * 10 + j * 3 + i) for i, (n, k) in enumerate(shapes)]
        packed, w_scale = bl.pack_stacked([W.cuda() for W in Ws])
        g_layer[name], g_layer[name + "_scale"] = packed, w_scale
        qs, scales = [], []
        for W in Ws:
            _, gamma, q = oracle.pack_weights(W.numpy())
            qs.append(q)
            scales.append(np.full(W.shape[0], float(gamma)))
        o_layer[name] = np.concatenate(qs)
        o_layer[name + "_scale"] = np.concatenate(scales)
    for j, (name, k) in enumerate({"gain_qkv": H, "gain_o": H, "gain_gate_up": H, "gain_down": F}.items()):
        g = synth.rms_gains(k, seed=seed * 10 + 7 + j)
        g_layer[name] = g.cuda()
        o_layer[name] = synth.bf16_bits(g)
    return g_layer, o_layer


@pytest.fixture(scope="module")
def layers():
    return [make_layer(H, NQKV, F, seed=100 + l) for l in range(2)]


def bitlinear_ref(in_bits, gain_bits, wq, w_scale, gpu_xq, gpu_sc, rows):
    """The oracle's BitLinear on the GPU's input: checks the codes and scales of every
    token, returns the fp64 outputs of the sampled tokens."""
    oq, osig = oracle.act_quant(in_bits, gain_bits, RMS_EPS)
    assert (gpu_xq == oq).all()
    assert np.all(np.abs(gpu_sc.astype(np.float64) - osig) <= SIGMA_RTOL * osig)
    acc = oracle.ternary_matmul(oq[rows], wq)
    return oracle.dequant(acc, osig[rows], w_scale)


def check_residual(gpu_bits, x_bits, y64):
    """gpu = bf16(fl32(x + y_gpu)) against the exact x + y (see the module docstring)."""
    g = oracle.bf16_bits_to_f64(gpu_bits)
    x = oracle.bf16_bits_to_f64(x_bits)
    exact = x + y64
    bound = 2.0 ** -8 * np.abs(exact) + 2.0 ** -24 * (np.abs(exact) + Y_RTOL * np.abs(y64)) + Y_RTOL * np.abs(y64)
    assert np.all(np.abs(g - exact) <= bound + 1e-38), float(np.max(np.abs(g - exact) - bound))


@pytest.mark.parametrize("M", [1, 8, 512])
def test_block_teacher_forced_per_bitlinear(layers, M):
    n = len(layers)
    x0 = synth.activations(M, H, seed=M, outliers=True)
    x = x0.cuda().clone()
    tb = bl.bitlinear_block_trace_bytes(M, H, NQKV, F)
    trace = torch.empty(n * tb + 256, dtype=torch.uint8, device="cuda")
    off = (-trace.data_ptr()) % 256
    trace = trace[off:off + n * tb]
    bl.bitlinear_block_forward([l[0] for l in layers], x, H, NQKV, F, RMS_EPS, flags=bl.FLAG_PDL, trace=trace)
    torch.cuda.synchronize()
    assert bl.bitlinear_get_device_error() == 0
    rows = np.arange(M) if M <= 8 else np.unique(np.concatenate(
        [[0, M - 1], np.random.default_rng(M).choice(M, 22, replace=False)]))
    x_in = synth.bf16_bits(x0)
    for li, (_, ol) in enumerate(layers):
        t = bl.block_trace_views(trace, li, M, H, NQKV, F)
        tn = {k: v.cpu() for k, v in t.items()}
        # QKV on the layer input
        y = bitlinear_ref(x_in, ol["gain_qkv"], ol["qkv"], ol["qkv_scale"], tn["xq_qkv"].numpy(),
                          tn["sc_qkv"].numpy(), rows)
        qkv_bits = bits(tn["qkv"])
        assert ulp_distance(qkv_bits[rows], oracle.f32_to_bf16_bits(y.astype(np.float32))).max() <= 1
        # O on the query slice, added to the residual stream
        q_bits = np.ascontiguousarray(qkv_bits[:, :H])
        y = bitlinear_ref(q_bits, ol["gain_o"], ol["o"], ol["o_scale"], tn["xq_o"].numpy(), tn["sc_o"].numpy(), rows)
        x_mid = bits(tn["x_mid"])
        check_residual(x_mid[rows], x_in[rows], y)
        # gate|up on the residual stream
        y = bitlinear_ref(x_mid, ol["gain_gate_up"], ol["gate_up"], ol["gate_up_scale"], tn["xq_gate_up"].numpy(),
                          tn["sc_gate_up"].numpy(), rows)
        gu = tn["gate_up"].numpy().astype(np.float64)
        assert np.all(np.abs(gu[rows] - y) <= F32_RTOL * np.abs(y))
        # down on h = bf16(relu(gate)^2 * up) of the GPU's gate|up, added to the residual
        gu32 = tn["gate_up"].numpy()
        h_bits = oracle.relu2_gate_bits(np.ascontiguousarray(gu32[:, :F]), np.ascontiguousarray(gu32[:, F:]))
        y = bitlinear_ref(h_bits, ol["gain_down"], ol["down"], ol["down_scale"], tn["xq_down"].numpy(),
                          tn["sc_down"].numpy(), rows)
        x_out = bits(tn["x_out"])
        check_residual(x_out[rows], x_mid[rows], y)
        x_in = x_out                          # the next layer's input, teacher forced
    assert (bits(x.cpu()) == x_in).all()      # the trace's last output is the block's output


def test_trace_changes_nothing(layers):
    M = 8
    x0 = synth.activations(M, H, seed=5).cuda()
    x1, x2 = x0.clone(), x0.clone()
    bl.bitlinear_block_forward([l[0] for l in layers], x1, H, NQKV, F, RMS_EPS, flags=bl.FLAG_PDL)
    trace = torch.empty(2 * bl.bitlinear_block_trace_bytes(M, H, NQKV, F) + 256, dtype=torch.uint8, device="cuda")
    off = (-trace.data_ptr()) % 256
    bl.bitlinear_block_forward([l[0] for l in layers], x2, H, NQKV, F, RMS_EPS, flags=bl.FLAG_PDL,
                               trace=trace[off:])
    torch.cuda.synchronize()
    assert torch.equal(x1, x2)


def test_block_forward_small_dims_two_layers_end_to_end():
    # a small stack end to end against oracle.block_layer: each layer's output within the
    # residual bound of one rounding, composed over two layers (no teacher forcing: an
    # intermediate within its bound can still move a code, so only the statistics of
    # exact agreement and the size of the differences are bounded)
    Hs, NQs, Fs = 256, 384, 512
    ls = [make_layer(Hs, NQs, Fs, seed=200 + l) for l in range(2)]
    for M in (1, 5, 40):
        x0 = synth.activations(M, Hs, seed=M)
        x = x0.cuda().clone()
        bl.bitlinear_block_forward([l[0] for l in ls], x, Hs, NQs, Fs, RMS_EPS, flags=bl.FLAG_PDL)
        torch.cuda.synchronize()
        o = oracle.block_layer(oracle.block_layer(synth.bf16_bits(x0), ls[0][1], RMS_EPS), ls[1][1], RMS_EPS)
        d = ulp_distance(bits(x.cpu()), o)
        assert (d == 0).mean() >= 0.98


def test_block_forward_zero_layers_and_errors():
    x = torch.zeros((2, 256), dtype=torch.bfloat16, device="cuda")
    assert bl.bitlinear_block_forward([], x, 256, 384, 512) is x
    layer, _ = make_layer(256, 384, 512, seed=3)
    with pytest.raises(bl.BitLinearError):
        bl.bitlinear_block_forward([layer], x, 256, 200, 512)       # NQKV < H
    with pytest.raises(bl.BitLinearError):                          # trace too small
        t = torch.empty(1024, dtype=torch.uint8, device="cuda")
        bl.bitlinear_block_forward([layer], x, 256, 384, 512, trace=t[(-t.data_ptr()) % 256:][:256])
