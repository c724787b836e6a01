"""GPU parity of bitlinear_block_forward (the BitLinear stack of transformer
layers) against oracle.block_layer.

Bars: one layer from the same input (teacher forced) must give bit-identical
bf16 outputs for at least 99.5% of the elements and differ by at most 2 bf16
ulp anywhere; two layers end to end at most 4 ulp.  Inside a layer the GPU
and the oracle round their BitLinear outputs to fp32 along different paths
(fl(fl(acc * sigma) * gamma) from a sigma within 4.5 fp32 ulp, against one
rounding of the fp64 value), so a value lying within a few fp32 ulp of a bf16
rounding boundary can round the other way; a changed bf16 input can then move
an int8 code of the next quantization by one, which moves that BitLinear's
output by one quantum.  Each BitLinear itself is checked bit-exactly by
test_gpu_parity.py.
"""
import numpy as np
import pytest
import torch

import bitlinear_rmsnorm_token_int8_b300 as bl
import oracle
from bitlinear_rmsnorm_token_int8_b300 import synth

pytestmark = pytest.mark.gpu

RMS_EPS = float(np.float32(1e-5))


def ulp_distance(a_bits, b_bits):
    def ordered(u):
        u = u.astype(np.int32)
        return np.where(u & 0x8000, -(u & 0x7FFF), u & 0x7FFF)
    return np.abs(ordered(a_bits) - ordered(b_bits))


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


@pytest.mark.parametrize("M", [1, 5, 40])
def test_block_forward_matches_oracle(M):
    H, NQKV, F = 256, 384, 512
    layers = [make_layer(H, NQKV, F, seed=100 + l) for l in range(2)]
    x0 = synth.activations(M, H, seed=M)
    x0_bits = synth.bf16_bits(x0)
    # one layer, teacher forced
    x = x0.cuda().clone()
    bl.bitlinear_block_forward([layers[0][0]], x, H, NQKV, F, RMS_EPS)
    torch.cuda.synchronize()
    assert bl.bitlinear_get_device_error() == 0
    g1 = synth.bf16_bits(x.cpu())
    o1 = oracle.block_layer(x0_bits, layers[0][1], RMS_EPS)
    d = ulp_distance(g1, o1)
    assert (d == 0).mean() >= 0.995 and d.max() <= 2, (float((d == 0).mean()), int(d.max()))
    # two layers end to end
    x = x0.cuda().clone()
    bl.bitlinear_block_forward([l[0] for l in layers], x, H, NQKV, F, RMS_EPS, flags=bl.FLAG_PDL)
    torch.cuda.synchronize()
    o2 = oracle.block_layer(o1, layers[1][1], RMS_EPS)
    assert ulp_distance(synth.bf16_bits(x.cpu()), o2).max() <= 4


def test_block_forward_many_rows():
    # M = 320 runs the prefill contraction on every projection.  A
    # teacher-forced layer is four quantizations deep: an intermediate bf16 value that
    # is 1 ulp from the oracle's (allowed) can flip one int8 code of the next
    # quantization, which moves that row's outputs by about one code's worth,
    # gamma * sigma per unit weight: a few rows differ by more than 2 ulp, by a small
    # amount against the outputs' scale.  Bar: >= 99 % identical, every difference
    # below 5 % of the RMS of the layer output.
    M, H, NQKV, F = 320, 256, 384, 512
    layer, olayer = make_layer(H, NQKV, F, seed=100)
    x0 = synth.activations(M, H, seed=M)
    x = x0.cuda().clone()
    bl.bitlinear_block_forward([layer], x, H, NQKV, F, RMS_EPS)
    torch.cuda.synchronize()
    assert bl.bitlinear_get_device_error() == 0
    g = synth.bf16_bits(x.cpu())
    o = oracle.block_layer(synth.bf16_bits(x0), olayer, RMS_EPS)
    assert (ulp_distance(g, o) == 0).mean() >= 0.99
    gf = x.cpu().float().numpy().astype(np.float64)
    of = torch.from_numpy(o.view(np.int16)).view(torch.bfloat16).float().numpy().astype(np.float64)
    assert np.abs(gf - of).max() <= 0.05 * np.sqrt(np.mean(of ** 2))


def test_block_forward_zero_layers_and_errors():
    x = torch.zeros((2, 256), dtype=torch.bfloat16, device="cuda")
    assert bl.bitlinear_block_forward([], x, 256, 384, 512) is x
    layer, _ = make_layer(256, 384, 512, seed=3)
    with pytest.raises(bl.BitLinearError):
        bl.bitlinear_block_forward([layer], x, 256, 200, 512)       # NQKV < H
