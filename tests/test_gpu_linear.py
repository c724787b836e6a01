"""GPU parity of bitlinear_linear_forward, the whole BitLinear layer in one call
(RMSNorm + absmax int8 quantization + ternary contraction + dequantization),
against the CPU oracle, on the decode (M <= 32) and prefill routes.  Same bars as
test_gpu_parity.py: codes and accumulators bit-exact, act_scale within 5e-7,
fp32 y within 1e-6 relative, bf16 y within 1 ulp."""
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


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    bl.lib()
    yield
    assert bl.bitlinear_get_device_error() == 0


def bf16_ulp_distance(a_bits, b_bits):
    def ordered(u):
        u = u.astype(np.int32)
        return np.where(u & 0x8000, -(u & 0x7FFF), u & 0x7FFF)
    return np.abs(ordered(a_bits) - ordered(b_bits))


def check_y(y: torch.Tensor, o_y: np.ndarray):
    if y.dtype == torch.float32:
        g = y.cpu().numpy().astype(np.float64)
        assert np.all(np.abs(g - o_y) <= F32_RTOL * np.abs(o_y))
    else:
        gb = y.cpu().view(torch.int16).numpy().view(np.uint16)
        ob = oracle.f32_to_bf16_bits(o_y.astype(np.float32))
        assert bf16_ulp_distance(gb, ob).max() <= 1


def run_linear(M, N, K, dt, seed, gain=True, rms_eps=RMS_EPS, flags=0, outliers=True):
    x = synth.activations(M, K, seed=seed, outliers=outliers)
    g = synth.rms_gains(K, seed=seed + 1) if gain else None
    W = synth.latent_weights(N, K, seed=seed + 2)
    packed, w_scale, gamma = bl.bitlinear_pack_weights(W.cuda())
    xq = torch.empty((M, K), dtype=torch.int8, device="cuda")
    sc = torch.empty(M + 3, dtype=torch.float32, device="cuda")[:M]
    acc = torch.empty((M, N), dtype=torch.int32, device="cuda")
    y = bl.bitlinear_linear_forward(x.cuda(), None if g is None else g.cuda(), rms_eps, packed, w_scale,
                                    out_dtype=dt, x_q=xq, act_scale=sc, acc_debug=acc, flags=flags)
    torch.cuda.synchronize()
    o_xq, o_sig = oracle.act_quant(synth.bf16_bits(x), None if g is None else synth.bf16_bits(g), rms_eps)
    _, o_gamma, o_wq = oracle.pack_weights(W.numpy())
    assert float(gamma.cpu().item()) == float(o_gamma)
    assert (xq.cpu().numpy() == o_xq).all()
    assert np.all(np.abs(sc.cpu().numpy().astype(np.float64) - o_sig) <= SIGMA_RTOL * o_sig)
    o_acc = oracle.ternary_matmul(o_xq, o_wq)
    assert (acc.cpu().numpy() == o_acc).all()
    check_y(y, oracle.dequant(o_acc, o_sig, np.full(N, float(o_gamma))))
    return dict(x=x, g=g, packed=packed, w_scale=w_scale, y=y, acc=acc, xq=xq, sc=sc)


@pytest.mark.parametrize("M,N,K,dt", [
    (1, 2560, 2560, torch.bfloat16),     # one segment per CTA, clusters of 5
    (1, 144, 1152, torch.float32),       # ragged K slices (3 segments over the cluster)
    (4, 512, 256, torch.float32),        # half a segment of zero-padded K
    (8, 3840, 2560, torch.bfloat16),
    (8, 2560, 6912, torch.bfloat16),     # K = 13.5 segments: the last slice ends inside a segment
    (11, 400, 4608, torch.float32),      # 11 tokens: two 8-token groups, the second ragged
    (16, 1040, 4096, torch.bfloat16),
    (3, 272, 14336, torch.float32),      # longest K: partial sums up to 127 * 14336
])
def test_linear_decode_matches_oracle(M, N, K, dt):
    run_linear(M, N, K, dt, seed=31 * M + N + K)


@pytest.mark.parametrize("M,N,K", [(17, 160, 1024), (40, 256, 2560), (300, 384, 512)])
def test_linear_more_tokens_matches_oracle(M, N, K):
    run_linear(M, N, K, torch.float32, seed=7 * M + N + K)


def test_linear_without_gain_and_without_rmsnorm():
    run_linear(5, 512, 1024, torch.float32, seed=501, gain=False)
    run_linear(5, 512, 1024, torch.float32, seed=502, rms_eps=-1.0)


def test_linear_every_small_m():
    for M in range(1, 17):
        run_linear(M, 144, 1536, torch.float32, seed=700 + M)


def test_linear_equals_quant_then_forward():
    # one call and the two calls give the same codes, accumulators and outputs
    for M, N, K in [(1, 2560, 2560), (8, 13824, 2560), (16, 2560, 6912)]:
        x = synth.activations(M, K, seed=M + K).cuda()
        g = synth.rms_gains(K, seed=K).cuda()
        W = synth.latent_weights(N, K, seed=N).cuda()
        packed, w_scale, _ = bl.bitlinear_pack_weights(W)
        acc1 = torch.empty((M, N), dtype=torch.int32, device="cuda")
        xq1 = torch.empty((M, K), dtype=torch.int8, device="cuda")
        y1 = bl.bitlinear_linear_forward(x, g, RMS_EPS, packed, w_scale, out_dtype=torch.float32,
                                         x_q=xq1, acc_debug=acc1)
        xq2, sc2 = bl.bitlinear_quant_act(x, g, RMS_EPS)
        acc2 = torch.empty((M, N), dtype=torch.int32, device="cuda")
        y2 = bl.bitlinear_forward(xq2, sc2, packed, w_scale, out_dtype=torch.float32, acc_debug=acc2)
        torch.cuda.synchronize()
        assert torch.equal(xq1, xq2) and torch.equal(acc1, acc2) and torch.equal(y1, y2)


@pytest.mark.parametrize("M", [1, 2, 8])
def test_linear_residual_and_pdl_chain(M):
    # two layers back to back with programmatic dependent launch: the second reads the
    # first's bf16 output (written by the kernel it overlaps with), then adds into a
    # residual; one and two tokens run on the int8-code kernel, eight on the tensor cores
    H = 2048
    x = synth.activations(M, H, seed=91)
    g = synth.rms_gains(H, seed=92)
    W1 = synth.latent_weights(H, H, seed=93)
    W2 = synth.latent_weights(H, H, seed=94)
    p1, s1, g1 = bl.bitlinear_pack_weights(W1.cuda())
    p2, s2, g2 = bl.bitlinear_pack_weights(W2.cuda())
    r0 = synth.activations(M, H, seed=95, outliers=False)
    res = r0.cuda().clone()
    h = bl.bitlinear_linear_forward(x.cuda(), g.cuda(), RMS_EPS, p1, s1, out_dtype=torch.bfloat16,
                                    flags=bl.FLAG_PDL)
    bl.bitlinear_linear_forward(h, g.cuda(), RMS_EPS, p2, s2, out_dtype=torch.bfloat16, y=res,
                                residual=True, flags=bl.FLAG_PDL)
    torch.cuda.synchronize()
    gb = synth.bf16_bits(g)
    o_xq, o_sig = oracle.act_quant(synth.bf16_bits(x), gb, RMS_EPS)
    _, o_g1, o_w1 = oracle.pack_weights(W1.numpy())
    o_h = oracle.dequant(oracle.ternary_matmul(o_xq, o_w1), o_sig, np.full(H, float(o_g1)))
    hb = h.cpu().view(torch.int16).numpy().view(np.uint16)
    assert bf16_ulp_distance(hb, oracle.f32_to_bf16_bits(o_h.astype(np.float32))).max() <= 1
    # second layer from the GPU's own h (a 1-ulp difference in h would change codes)
    o_xq2, o_sig2 = oracle.act_quant(hb, gb, RMS_EPS)
    _, o_g2, o_w2 = oracle.pack_weights(W2.numpy())
    o_y2 = oracle.dequant(oracle.ternary_matmul(o_xq2, o_w2), o_sig2, np.full(H, float(o_g2)))
    r0f = r0.float().numpy().astype(np.float64)
    # y = bf16(fl32(r0) + result): within one bf16 ulp of the larger addend (the sum may cancel)
    got = res.cpu().float().numpy().astype(np.float64)
    scale = np.maximum(np.abs(r0f), np.abs(o_y2))
    assert np.all(np.abs(got - (r0f + o_y2)) <= 2.0 ** -7 * scale + 1e-30)


@pytest.mark.parametrize("M,K,N,gain,rms", [
    (1, 128, 144, True, True), (1, 1152, 272, False, True), (1, 2560, 3840, True, True),
    (1, 6912, 2560, True, False), (1, 8192, 400, True, True), (1, 4096, 28672, True, True),
    (1, 2560, 13824, False, True),
    # K above 8192 (matrices of at least 12 MiB): two of the quantization's threads per thread
    (1, 14336, 4096, True, True), (1, 10240, 5120, True, False), (1, 16384, 3200, False, True)])
def test_linear_one_token_fused(M, K, N, gain, rms):
    # one token: RMSNorm, quantization and the contraction in one kernel.
    # Its codes, scales, accumulators and outputs equal the oracle's and, bit for bit, those
    # of the two-kernel path (quantization, then the contraction on the int8 codes)
    assert bl.bitlinear_linear_route(M, N, K) == bl.ROUTE_FUSED
    eps = RMS_EPS if rms else -1.0
    r = run_linear(M, N, K, torch.float32, seed=K + N + M, gain=gain, rms_eps=eps, flags=bl.FLAG_PDL)
    xq2, sc2 = bl.bitlinear_quant_act(r["x"].cuda(), None if r["g"] is None else r["g"].cuda(), eps)
    acc2 = torch.empty((M, N), dtype=torch.int32, device="cuda")
    y2 = bl.bitlinear_forward(xq2, sc2, r["packed"], r["w_scale"], out_dtype=torch.float32, acc_debug=acc2)
    torch.cuda.synchronize()
    assert torch.equal(r["xq"], xq2) and torch.equal(r["sc"], sc2)
    assert torch.equal(r["acc"], acc2) and torch.equal(r["y"], y2)


@pytest.mark.parametrize("M,N,K", [
    (1, 2560, 2560),      # the one-kernel layer
    (1, 4096, 14336),     # quantization + the int8-code kernel
    (2, 3840, 2560),      # two tokens on the int8-code kernel
    (8, 3840, 2560),      # quantization + tcgen05 decode
    (16, 1040, 4096),
    (64, 512, 1536),      # prefill (takes no prefetch)
])
def test_l2_prefetch_hint_changes_nothing(M, N, K):
    # the l2_prefetch range (here the packed weights of a second matrix, as in a chain of
    # calls) is a cache hint: codes, accumulators and outputs are bit-identical with it
    x = synth.activations(M, K, seed=M + N).cuda()
    g = synth.rms_gains(K, seed=K).cuda()
    packed, w_scale, _ = bl.bitlinear_pack_weights(synth.latent_weights(N, K, seed=N).cuda())
    nxt, _, _ = bl.bitlinear_pack_weights(synth.latent_weights(2 * N, K, seed=N + 1).cuda())
    outs = []
    for pf in (None, nxt, (nxt, 1000)):
        acc = torch.empty((M, N), dtype=torch.int32, device="cuda")
        y = bl.bitlinear_linear_forward(x, g, RMS_EPS, packed, w_scale, out_dtype=torch.float32, acc_debug=acc,
                                        flags=bl.FLAG_PDL, prefetch=pf)
        xq, sc = bl.bitlinear_quant_act(x, g, RMS_EPS)
        acc2 = torch.empty((M, N), dtype=torch.int32, device="cuda")
        y2 = bl.bitlinear_forward(xq, sc, packed, w_scale, out_dtype=torch.float32, acc_debug=acc2, prefetch=pf)
        torch.cuda.synchronize()
        outs.append((y.cpu(), acc.cpu(), y2.cpu(), acc2.cpu()))
    for o in outs[1:]:
        for a, b in zip(outs[0], o):
            assert torch.equal(a, b)
    assert torch.equal(outs[0][1], outs[0][3])


def test_prefill_cluster_size_by_memory_kind():
    # clusters of two (one multicast copy of each activation block for both CTAs) only
    # for operands in this device's own memory
    d = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    assert bl.bitlinear_prefill_cluster_size(d, 2048, 14336, 4096) == 2
    assert bl.bitlinear_prefill_cluster_size(d, 2048, 128, 4096) == 1      # one weight block
    assert bl.bitlinear_prefill_cluster_size(d, 16, 14336, 4096) == -1     # decode route
    pinned = torch.empty(1 << 20, dtype=torch.uint8, pin_memory=True)
    assert bl.bitlinear_prefill_cluster_size(pinned, 2048, 14336, 4096) == 1
    pageable = torch.empty(1 << 20, dtype=torch.uint8)
    assert bl.bitlinear_prefill_cluster_size(pageable, 2048, 14336, 4096) == 1
