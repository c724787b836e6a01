"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle on the
same seeded inputs.

Bars:
* int8 codes, packed bytes, gamma and int32 accumulators: bit-exact;
* act_scale (sigma): relative error <= 5e-7 against the oracle's fp64 value (the
  GPU sums x^2 as an error-free fp32 pair, then takes five IEEE-rounded steps:
  at most 4.5 * 2^-24 = 2.7e-7);
* fp32 output: relative error <= 1e-6 against the oracle's fp64 output (sigma's
  error plus two fp32 roundings: at most 3.9e-7);
* bf16 output: within 1 bf16 ulp of the oracle's fp64 output rounded to bf16 (the
  fp32 value is that close to the exact one).
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

RMS_EPS = float(np.float32(1e-5))
SIGMA_RTOL = 5e-7
F32_RTOL = 1e-6


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    bl.lib()
    yield
    assert bl.bitlinear_get_device_error() == 0


def bf16_ulp_distance(a_bits: np.ndarray, b_bits: np.ndarray) -> np.ndarray:
    def ordered(u):
        u = u.astype(np.int32)
        return np.where(u & 0x8000, -(u & 0x7FFF), u & 0x7FFF)
    return np.abs(ordered(a_bits) - ordered(b_bits))


def f64_to_bf16_bits(y: np.ndarray) -> np.ndarray:
    # round the fp64 value to fp32 then bf16; the double rounding can differ from a
    # direct fp64 -> bf16 rounding only at exact bf16 ties, within the 1-ulp bar
    return oracle.f32_to_bf16_bits(y.astype(np.float32))


def gpu_quant(x_bf16: torch.Tensor, gain, rms_eps):
    xq, sc = bl.bitlinear_quant_act(x_bf16.cuda(), None if gain is None else gain.cuda(), rms_eps)
    torch.cuda.synchronize()
    return xq.cpu().numpy(), sc.cpu().numpy().astype(np.float64)


def gpu_pack(W: torch.Tensor, eps=1e-5):
    """GPU packing; the packed bytes come back in the canonical [N, K/4] order."""
    N, K = W.shape
    packed, ws, gamma = bl.bitlinear_pack_weights(W.cuda(), eps)
    torch.cuda.synchronize()
    tiled = packed.cpu().numpy()
    # the padding of the tiled layout (rows >= N, codes >= K) holds zero codes
    canon = layout.canonical_from_tiled(tiled, N, K)
    mask = np.ones(tiled.size, dtype=bool)
    mask[layout.packed_index(N, K)] = False
    assert not tiled[: layout.packed_bytes(N, K)][mask[: layout.packed_bytes(N, K)]].any()
    return canon, ws.cpu().numpy(), np.float32(gamma.cpu().item())


def tiled_cuda(canon: torch.Tensor, K: int) -> torch.Tensor:
    """Canonical [N, K/4] packed codes -> the tiled layout on the GPU."""
    return torch.from_numpy(layout.tiled_from_canonical(canon.numpy(), K)).cuda()


# ---------------------------------------------------------------------------
# activation quantization
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("M,K,gain,rms,outliers", [
    (1, 8, False, True, False), (3, 256, True, True, True), (17, 2560, True, True, True),
    (5, 6912, False, True, True), (4, 14336, True, True, False), (2, 16392, True, True, True),
    (2, 65536, True, True, True), (33, 4096, True, False, True), (64, 1024, False, False, False),
])
def test_quant_act_matches_oracle(M, K, gain, rms, outliers):
    x = synth.activations(M, K, seed=10 * M + K, outliers=outliers)
    g = synth.rms_gains(K, seed=K) if gain else None
    eps = RMS_EPS if rms else -1.0
    xq, sc = gpu_quant(x, g, eps)
    oq, osig = oracle.act_quant(synth.bf16_bits(x), None if g is None else synth.bf16_bits(g), eps)
    assert (xq == oq).all()
    assert np.all(np.abs(sc - osig) <= SIGMA_RTOL * osig)


@pytest.mark.parametrize("M,K,gain,rms", [(600, 4104, True, True), (640, 6912, False, True), (700, 8192, True, False),
                                          (33, 2560, True, True), (2048, 4096, True, True), (300, 14336, False, True),
                                          (97, 65536, True, True)])
def test_quant_act_many_rows_matches_oracle(M, K, gain, rms):
    # many rows: one CTA per row, or for M >= 4 x the SM count and K > 4096 persistent
    # CTAs streaming rows through shared memory; K = 4104 ends in half a 16-input unit
    x = synth.activations(M, K, seed=M + 3 * K)
    g = synth.rms_gains(K, seed=K + 1) if gain else None
    eps = RMS_EPS if rms else -1.0
    xq, sc = gpu_quant(x, g, eps)
    oq, osig = oracle.act_quant(synth.bf16_bits(x), None if g is None else synth.bf16_bits(g), eps)
    assert (xq == oq).all()
    assert np.all(np.abs(sc - osig) <= SIGMA_RTOL * osig)


def test_quant_act_edge_rows():
    K = 512
    rows = np.zeros((6, K), dtype=np.float32)
    rows[1, 0] = 127.0                         # ties: 127 * x / 127 = x
    rows[1, 1:9] = [2.5, 1.5, 0.5, -0.5, -1.5, -2.5, 3.5, -3.5]
    rows[2, :] = 1e-12                         # max below the 1e-8 guard
    rows[2, 7] = -3e-12
    rows[3, :] = -7.0                          # constant row
    rng = np.random.default_rng(0)
    rows[4] = rng.integers(-254, 255, K) / 2.0  # many half-integer ties after scaling
    rows[4, 3] = 127.0
    rows[5] = rng.standard_normal(K) * 1e15     # large magnitudes (|x| <= 2^60 contract)
    bits = oracle.f32_to_bf16_bits(rows)
    x = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16)
    for gain in (None, synth.rms_gains(K, seed=3)):
        xq, sc = gpu_quant(x, gain, RMS_EPS)
        oq, osig = oracle.act_quant(bits, None if gain is None else synth.bf16_bits(gain), RMS_EPS)
        assert (xq == oq).all()
        assert np.all(np.abs(sc - osig) <= SIGMA_RTOL * osig)
    assert (xq[0] == 0).all()


_GOLDEN = json.load(open(os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "worked_examples.json")))


@pytest.mark.parametrize("key", ["act_clamp_regular_tiny_row", "act_clamp_plain_tiny_row",
                                 "act_clamp_small_rmsnorm_row"])
@pytest.mark.parametrize("kernel", ["one_row_per_cta", "many_rows", "one_token_layer", "one_token_layer_long"])
def test_quant_clamp_golden_rows_every_kernel(key, kernel):
    # activation_quant clamps the max of the RMSNorm output at 1e-8: the hand-worked rows
    # (zero-padded, which changes neither max|n| nor the rounding of mean(x^2) + eps)
    # through each kernel that quantizes
    ex = _GOLDEN[key]
    eps = RMS_EPS if ex["rms_eps"] >= 0 else -1.0
    K = {"many_rows": 4104, "one_token_layer_long": 14336}.get(kernel, 512)
    M = 600 if kernel == "many_rows" else 1
    rows = np.zeros((M, K), dtype=np.float32)
    rows[:, :8] = ex["x"]
    bits = oracle.f32_to_bf16_bits(rows)
    x = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16)
    want = np.zeros((M, K), dtype=np.int8)
    want[:, :8] = ex["x_q"]
    if kernel.startswith("one_token_layer"):
        N = 4096 if kernel == "one_token_layer_long" else 128    # the persistent kernel, two threads' units each
        assert bl.bitlinear_linear_route(1, N, K) == bl.ROUTE_FUSED
        packed, w_scale, _ = bl.bitlinear_pack_weights(synth.latent_weights(N, K, seed=5).cuda())
        xq = torch.empty((1, K), dtype=torch.int8, device="cuda")
        sc = torch.empty(4, dtype=torch.float32, device="cuda")[:1]
        bl.bitlinear_linear_forward(x.cuda(), None, eps, packed, w_scale, out_dtype=torch.float32, x_q=xq,
                                    act_scale=sc)
        torch.cuda.synchronize()
        xq, sc = xq.cpu().numpy(), sc.cpu().numpy().astype(np.float64)
    else:
        xq, sc = gpu_quant(x, None, eps)
    oq, osig = oracle.act_quant(bits, None, eps)
    assert (oq == want).all()
    assert (xq == want).all()
    assert np.all(np.abs(sc - osig) <= SIGMA_RTOL * osig)


def test_quant_act_empty_is_noop():
    x = torch.zeros((0, 256), dtype=torch.bfloat16, device="cuda")
    xq, sc = bl.bitlinear_quant_act(x)
    assert xq.shape == (0, 256) and sc.shape == (0,)


# ---------------------------------------------------------------------------
# weight packing
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("N,K", [(1, 4), (3, 20), (16, 256), (512, 256), (37, 2560), (2560, 6912)])
def test_pack_matches_oracle(N, K):
    W = synth.latent_weights(N, K, seed=N * 7 + K)
    packed, ws, gamma = gpu_pack(W)
    o_packed, o_gamma, _ = oracle.pack_weights(W.numpy())
    assert gamma == o_gamma
    assert (ws == o_gamma).all()
    assert (packed == o_packed).all()


def test_pack_adversarial_values():
    rng = np.random.default_rng(1)
    N, K = 24, 64
    W = (rng.standard_normal((N, K)) * np.exp2(rng.integers(-140, 60, (N, K)))).astype(np.float32)
    W[0, :8] = [1.4e-45, -1.4e-45, 1e-40, -0.0, 0.0, 3e38, -3e38, 1.0]
    for Wt in (W, np.abs(W), np.full((N, K), 2.0**-149, dtype=np.float32)):
        packed, ws, gamma = gpu_pack(torch.from_numpy(np.ascontiguousarray(Wt)))
        o_packed, o_gamma, _ = oracle.pack_weights(Wt)
        assert gamma == o_gamma, (gamma, o_gamma)
        assert (packed == o_packed).all()


def test_pack_gamma_ties_round_to_even():
    # mean = 1 + 2^-24 exactly: halfway between 1 and 1 + 2^-23 -> 1 (even)
    # mean = 1 + 3*2^-24: halfway between 1 + 2^-23 (odd) and 1 + 2^-22 -> 1 + 2^-22
    one_up = np.float32(1 + 2.0**-23)
    for w, expect in (([1.0, one_up, 1.0, one_up], np.float32(1.0)),
                      ([one_up, np.float32(1 + 2.0**-22), one_up, np.float32(1 + 2.0**-22)],
                       np.float32(1 + 2.0**-22))):
        Wt = torch.tensor([w], dtype=torch.float32)
        _, _, gamma = gpu_pack(Wt)
        assert gamma == expect == oracle.absmean_gamma(Wt.numpy())


def test_pack_threshold_ties():
    # weights exactly at d/2 (a tie, rounds to 0) and one binary32 step above (rounds to 1)
    rng = np.random.default_rng(2)
    W = (rng.standard_normal((8, 64)) * 0.02).astype(np.float32)
    g = oracle.absmean_gamma(W)
    d = np.float32(g + np.float32(1e-5))
    half = np.float32(d / np.float32(2))
    # small edits that keep the absmean unchanged are hard; instead check codes with the
    # oracle on the full matrix including elements placed near the threshold
    W[0, :4] = [half, -half, np.nextafter(half, np.float32(1)), -np.nextafter(half, np.float32(1))]
    packed, _, gamma = gpu_pack(torch.from_numpy(W))
    o_packed, o_gamma, q = oracle.pack_weights(W)
    assert gamma == o_gamma and (packed == o_packed).all()


def test_pack_nonfinite_sets_device_error():
    W = torch.zeros((4, 16), dtype=torch.float32)
    W[1, 3] = float("inf")
    bl.bitlinear_pack_weights(W.cuda())
    assert bl.bitlinear_get_device_error() == 9
    assert bl.bitlinear_get_device_error() == 0


# ---------------------------------------------------------------------------
# contraction + dequantization
# ---------------------------------------------------------------------------

def run_forward(M, N, K, out_dtype, seed, outliers=True, gain=True):
    x = synth.activations(M, K, seed=seed, outliers=outliers)
    g = synth.rms_gains(K, seed=seed + 1) if gain else None
    W = synth.latent_weights(N, K, seed=seed + 2)
    packed, w_scale, gamma = bl.bitlinear_pack_weights(W.cuda())
    xq, sc = bl.bitlinear_quant_act(x.cuda(), None if g is None else g.cuda(), RMS_EPS)
    acc = torch.empty((M, N), dtype=torch.int32, device="cuda")
    y = bl.bitlinear_forward(xq, sc, packed, w_scale, out_dtype=out_dtype, acc_debug=acc)
    torch.cuda.synchronize()
    o_xq, o_sig = oracle.act_quant(synth.bf16_bits(x), None if g is None else synth.bf16_bits(g), RMS_EPS)
    o_packed, o_gamma, o_wq = oracle.pack_weights(W.numpy())
    return dict(x=x, y=y.cpu(), acc=acc.cpu().numpy(), xq=xq.cpu().numpy(), sc=sc.cpu().numpy(),
                packed=layout.canonical_from_tiled(packed.cpu().numpy(), N, K),
                gamma=np.float32(gamma.cpu().item()),
                o_xq=o_xq, o_sig=o_sig, o_packed=o_packed, o_gamma=o_gamma, o_wq=o_wq)


def check_output(r, ts=None, ns=None):
    """acc bit-exact; y against the oracle's fp64 y (all, or at (ts, ns))."""
    assert (r["xq"] == r["o_xq"]).all()
    assert (r["packed"] == r["o_packed"]).all() and r["gamma"] == r["o_gamma"]
    if ts is None:
        o_acc = oracle.ternary_matmul(r["o_xq"], r["o_wq"])
        assert (r["acc"] == o_acc).all()
        N = o_acc.shape[1]
        o_y = oracle.dequant(o_acc, r["o_sig"], np.full(N, float(r["o_gamma"])))
        gy = r["y"]
    else:
        o_acc = oracle.ternary_matmul_at(r["o_xq"], r["o_wq"], ts, ns)
        assert (r["acc"][ts, ns] == o_acc).all()
        o_y = o_acc.astype(np.float64) * r["o_sig"][ts] * float(r["o_gamma"])
        gy = r["y"][ts, ns]
    if gy.dtype == torch.float32:
        g = gy.numpy().astype(np.float64)
        assert np.all(np.abs(g - o_y) <= F32_RTOL * np.abs(o_y))
    else:
        gb = gy.view(torch.int16).numpy().view(np.uint16)
        assert bf16_ulp_distance(gb, f64_to_bf16_bits(o_y)).max() <= 1


@pytest.mark.parametrize("M,N,K,dt", [
    (4, 512, 256, torch.float32),        # the single-layer K=256 -> N=512, 4-token case
    (1, 16, 128, torch.float32), (3, 48, 384, torch.bfloat16), (8, 272, 640, torch.float32),
    (17, 160, 1024, torch.bfloat16), (16, 2560, 2560, torch.float32), (40, 256, 6912, torch.bfloat16),
    (129, 384, 512, torch.float32),
    (24, 272, 4608, torch.bfloat16),     # three 8-token groups, K split over a cluster of CTAs
    (32, 400, 1536, torch.float32),      # the largest decode M; a partial 128-row tile
])
def test_forward_matches_oracle(M, N, K, dt):
    r = run_forward(M, N, K, dt, seed=M * 131 + N + K)
    check_output(r)


@pytest.mark.parametrize("M,K", [(1, 128), (1, 640), (2, 640), (1, 4096), (2, 4096), (1, 6912), (1, 14336),
                                 (1, 65536), (2, 14336), (2, 37376)])
def test_codes_route_equals_operand_route(M, K):
    # one or two tokens given x_q run on the int8-code (CUDA-core) kernel; given only the
    # operand form, on the tensor cores: same accumulators and outputs, both equal to the
    # oracle's (N = 272: a second weight tile of 16 rows)
    N = 272
    x = synth.activations(M, K, seed=M + K)
    W = synth.latent_weights(N, K, seed=K + 3)
    packed, w_scale, gamma = bl.bitlinear_pack_weights(W.cuda())
    xq, sc, ops = bl.bitlinear_quant_act(x.cuda(), None, RMS_EPS, x_ops=True)
    assert bl.bitlinear_forward_workspace_bytes(M, N, K) == 0          # the codes route needs none
    for dt in (torch.float32, torch.bfloat16):
        acc1 = torch.empty((M, N), dtype=torch.int32, device="cuda")
        acc2 = torch.empty((M, N), dtype=torch.int32, device="cuda")
        y1 = bl.bitlinear_forward(xq, sc, packed, w_scale, out_dtype=dt, acc_debug=acc1, flags=bl.FLAG_PDL)
        y2 = bl.bitlinear_forward(None, sc, packed, w_scale, out_dtype=dt, acc_debug=acc2, x_ops=ops, K=K)
        torch.cuda.synchronize()
        assert torch.equal(acc1, acc2) and torch.equal(y1, y2)
    o_xq, _ = oracle.act_quant(synth.bf16_bits(x), None, RMS_EPS)
    _, _, o_wq = oracle.pack_weights(W.numpy())
    assert (xq.cpu().numpy() == o_xq).all()
    assert (acc1.cpu().numpy() == oracle.ternary_matmul(o_xq, o_wq)).all()


@pytest.mark.parametrize("M,K,N", [(1, 14336, 4096), (2, 4096, 28672), (2, 14336, 4096), (1, 65536, 2048),
                                   (2, 37376, 1408)])
def test_codes_route_large_matrices(M, K, N):
    # from 12 MiB of packed weights the int8-code route runs the persistent CUDA-core
    # kernel (one CTA per SM, weights streamed through shared memory): same accumulators
    # and outputs as the tensor cores on the operand form, and as the oracle
    x = synth.activations(M, K, seed=7 * M + K)
    W = synth.latent_weights(N, K, seed=N + K)
    packed, w_scale, gamma = bl.bitlinear_pack_weights(W.cuda())
    assert bl.bitlinear_packed_bytes(N, K) >= 12 << 20
    xq, sc, ops = bl.bitlinear_quant_act(x.cuda(), None, RMS_EPS, x_ops=True)
    assert bl.bitlinear_forward_workspace_bytes(M, N, K) == 0
    acc1 = torch.empty((M, N), dtype=torch.int32, device="cuda")
    acc2 = torch.empty((M, N), dtype=torch.int32, device="cuda")
    y1 = bl.bitlinear_forward(xq, sc, packed, w_scale, out_dtype=torch.float32, acc_debug=acc1, flags=bl.FLAG_PDL)
    y2 = bl.bitlinear_forward(None, sc, packed, w_scale, out_dtype=torch.float32, acc_debug=acc2, x_ops=ops, K=K)
    torch.cuda.synchronize()
    assert torch.equal(acc1, acc2) and torch.equal(y1, y2)
    o_xq, _ = oracle.act_quant(synth.bf16_bits(x), None, RMS_EPS)
    _, _, o_wq = oracle.pack_weights(W.numpy())
    assert (xq.cpu().numpy() == o_xq).all()
    assert (acc1.cpu().numpy() == oracle.ternary_matmul(o_xq, o_wq)).all()


def test_forward_every_decode_m():
    # every token count the decode kernel takes (1..32: 8-token groups and their ragged ends)
    for M in range(1, 33):
        r = run_forward(M, 144, 1152, torch.float32, seed=9000 + M)
        check_output(r)


@pytest.mark.parametrize("M,N,K,dt,pdl", [
    (1, 2560, 2560, torch.bfloat16, True), (8, 3840, 2560, torch.bfloat16, True),
    (16, 4096, 4096, torch.bfloat16, False), (4, 512, 256, torch.float32, True),
    (5, 48, 384, torch.float32, True),           # K % 256 == 128: a half block at the end
    (17, 160, 640, torch.bfloat16, True),        # two 16-token tiles, the second ragged
    (2, 4096, 14336, torch.float32, False),      # largest K of the workloads, clusters of CTAs
])
def test_forward_from_quant_operands_matches_oracle(M, N, K, dt, pdl):
    # quant_act writes the tensor-core operand form, forward consumes it (no x_q read)
    flags = bl.FLAG_PDL if pdl else 0
    seed = M * 7 + N + K
    x = synth.activations(M, K, seed=seed)
    g = synth.rms_gains(K, seed=seed + 1)
    W = synth.latent_weights(N, K, seed=seed + 2)
    packed, w_scale, gamma = bl.bitlinear_pack_weights(W.cuda())
    xq, sc, ops = bl.bitlinear_quant_act(x.cuda(), g.cuda(), RMS_EPS, x_ops=True, flags=flags)
    acc = torch.empty((M, N), dtype=torch.int32, device="cuda")
    y = bl.bitlinear_forward(None, sc, packed, w_scale, out_dtype=dt, acc_debug=acc, x_ops=ops,
                             flags=flags, K=K)
    acc2 = torch.empty((M, N), dtype=torch.int32, device="cuda")
    y2 = bl.bitlinear_forward(xq, sc, packed, w_scale, out_dtype=dt, acc_debug=acc2, flags=flags)
    torch.cuda.synchronize()
    assert torch.equal(acc, acc2) and torch.equal(y, y2)     # both operand routes agree exactly
    o_xq, o_sig = oracle.act_quant(synth.bf16_bits(x), synth.bf16_bits(g), RMS_EPS)
    o_packed, o_gamma, o_wq = oracle.pack_weights(W.numpy())
    r = dict(y=y.cpu(), acc=acc.cpu().numpy(), xq=xq.cpu().numpy(),
             packed=layout.canonical_from_tiled(packed.cpu().numpy(), N, K),
             gamma=np.float32(gamma.cpu().item()), o_xq=o_xq, o_sig=o_sig, o_packed=o_packed,
             o_gamma=o_gamma, o_wq=o_wq)
    check_output(r)


@pytest.mark.parametrize("M,N,K,dt", [
    # 128-token tiles (few tiles: more of them fill more SMs)
    (33, 48, 512, torch.float32),       # just above the decode limit; one partial weight block
    (256, 160, 1024, torch.bfloat16),   # both halves of one operand block
    (300, 384, 2560, torch.float32),    # ragged third token tile
    (512, 256, 384, torch.bfloat16),    # K % 512 == 384: a zero-padded segment tail
    (80, 128, 14336, torch.float32),    # long K: |acc| up to 127 * 14336
    (600, 512, 1536, torch.bfloat16),   # five token tiles, the last one ragged and alone in its block
    # 256-token tiles (enough tiles for whole waves)
    (256, 19200, 512, torch.bfloat16),  # 75 cluster tiles on 74 clusters
    (300, 13824, 512, torch.float32),   # 108 cluster tiles, the second token tile ragged
    (38400, 128, 512, torch.bfloat16),  # one weight block: clusters of one, 150 tiles of 256 tokens
])
def test_prefill_matches_oracle(M, N, K, dt):
    # M > 32 tokens run on the tcgen05 kernel (weights decoded into tensor memory)
    for pdl in (0, bl.FLAG_PDL):
        seed = M + 3 * N + K + pdl
        x = synth.activations(M, K, seed=seed)
        g = synth.rms_gains(K, seed=seed + 1)
        W = synth.latent_weights(N, K, seed=seed + 2)
        packed, w_scale, gamma = bl.bitlinear_pack_weights(W.cuda())
        xq, sc, ops = bl.bitlinear_quant_act(x.cuda(), g.cuda(), RMS_EPS, x_ops=True, flags=pdl)
        acc = torch.empty((M, N), dtype=torch.int32, device="cuda")
        y = bl.bitlinear_forward(None, sc, packed, w_scale, out_dtype=dt, acc_debug=acc, x_ops=ops,
                                 flags=pdl, K=K)
        torch.cuda.synchronize()
        assert bl.bitlinear_get_device_error() == 0
        o_xq, o_sig = oracle.act_quant(synth.bf16_bits(x), synth.bf16_bits(g), RMS_EPS)
        o_packed, o_gamma, o_wq = oracle.pack_weights(W.numpy())
        r = dict(y=y.cpu(), acc=acc.cpu().numpy(), xq=xq.cpu().numpy(),
                 packed=layout.canonical_from_tiled(packed.cpu().numpy(), N, K),
                 gamma=np.float32(gamma.cpu().item()), o_xq=o_xq, o_sig=o_sig, o_packed=o_packed,
                 o_gamma=o_gamma, o_wq=o_wq)
        check_output(r)


@pytest.mark.parametrize("M,N,K,dt,rows,toks,step", [
    # 75 cluster tiles on 74 clusters: one cluster takes a second tile
    (256, 19200, 2048, torch.bfloat16, (18944, 19200), (0, 256), 1),
    # 94 cluster tiles: a partial second round of 20
    (256, 24064, 2048, torch.float32, (18944, 24064), (0, 256), 5),
    # 80 cluster tiles of 256 tokens, M = 500: the second round's 6 in the ragged token tile
    (500, 10240, 2048, torch.bfloat16, (8704, 10240), (256, 500), 3),
])
def test_prefill_partial_last_round_sampled(M, N, K, dt, rows, toks, step):
    # More cluster tiles than clusters: the persistent grid's partial last round;
    # every token of those tiles' rows (every step-th row) is compared, and a
    # random sample of the rest.
    seed = M + 5 * N + K
    x = synth.activations(M, K, seed=seed)
    g = synth.rms_gains(K, seed=seed + 1)
    W = synth.latent_weights(N, K, seed=seed + 2)
    packed, w_scale, gamma = bl.bitlinear_pack_weights(W.cuda())
    xq, sc, ops = bl.bitlinear_quant_act(x.cuda(), g.cuda(), RMS_EPS, x_ops=True, flags=bl.FLAG_PDL)
    acc = torch.empty((M, N), dtype=torch.int32, device="cuda")
    y = bl.bitlinear_forward(None, sc, packed, w_scale, out_dtype=dt, acc_debug=acc, x_ops=ops,
                             flags=bl.FLAG_PDL, K=K)
    torch.cuda.synchronize()
    assert bl.bitlinear_get_device_error() == 0
    o_xq, o_sig = oracle.act_quant(synth.bf16_bits(x), synth.bf16_bits(g), RMS_EPS)
    o_packed, o_gamma, o_wq = oracle.pack_weights(W.numpy())
    r = dict(y=y.cpu(), acc=acc.cpu().numpy(), xq=xq.cpu().numpy(),
             packed=layout.canonical_from_tiled(packed.cpu().numpy(), N, K),
             gamma=np.float32(gamma.cpu().item()), o_xq=o_xq, o_sig=o_sig, o_packed=o_packed,
             o_gamma=o_gamma, o_wq=o_wq)
    tt, nn = np.meshgrid(np.arange(*toks), np.arange(rows[0], rows[1], step), indexing="ij")
    rng = np.random.default_rng(seed)
    ts = np.concatenate([tt.ravel(), rng.integers(0, M, 4096), [0, M - 1]])
    ns = np.concatenate([nn.ravel(), rng.integers(0, N, 4096), [0, N - 1]])
    check_output(r, ts, ns)


def test_forward_exact_at_accumulator_extremes():
    # every partial sum at its largest magnitude: all codes +-127 against all-(+1) / all-(-1)
    # rows, and alternating signs so that partial sums swing between large values
    M, N, K = 16, 64, 14336
    xq = torch.full((M, K), 127, dtype=torch.int8)
    xq[1] = -127
    xq[2, ::2] = -127
    xq[3] = torch.randint(-127, 128, (K,), dtype=torch.int8)
    xq[4, : K // 2] = 127
    xq[4, K // 2:] = -127
    packed = torch.full((N, K // 4), 0x55, dtype=torch.uint8)
    packed[1::2] = 0xAA
    packed[2] = 0x66                       # codes 2,1,2,1: -1,+1,-1,+1 ... (byte 0b01100110)
    acc = torch.empty((M, N), dtype=torch.int32, device="cuda")
    bl.bitlinear_forward(xq.cuda(), torch.ones(M).cuda(), tiled_cuda(packed, K), torch.ones(N).cuda(),
                         out_dtype=torch.float32, acc_debug=acc)
    wq = oracle.unpack_codes(packed.numpy(), K)
    assert (acc.cpu().numpy() == oracle.ternary_matmul(xq.numpy(), wq)).all()


def test_forward_teacher_forced_dequant_is_two_roundings():
    # y = fl(fl(acc * sigma) * w_scale): with the GPU's own sigma and gamma the fp64
    # product differs from the fp32 output by at most two binary32 roundings
    r = run_forward(8, 512, 1024, torch.float32, seed=5)
    y64 = r["acc"].astype(np.float64) * r["sc"].astype(np.float64)[:, None] * float(r["gamma"])
    y32 = r["y"].numpy().astype(np.float64)
    assert np.all(np.abs(y32 - y64) <= 2.0**-23 * np.abs(y64))
    # and it is exactly that pair of fp32 products
    a = r["acc"].astype(np.float32) * r["sc"][:, None]
    assert (a.astype(np.float32) * r["gamma"] == r["y"].numpy()).all()


def test_forward_weight_invariants_on_gpu():
    # all +1 rows -> row sums of x_q; all -1 -> their negation; all 0 -> 0
    M, K = 5, 512
    xq = torch.randint(-127, 128, (M, K), dtype=torch.int8)
    sc = torch.ones(M, dtype=torch.float32)
    for code, sign in ((0x55, 1), (0xAA, -1), (0x00, 0)):
        packed = torch.full((32, K // 4), code, dtype=torch.uint8)
        acc = torch.empty((M, 32), dtype=torch.int32, device="cuda")
        bl.bitlinear_forward(xq.cuda(), sc.cuda(), tiled_cuda(packed, K), torch.ones(32).cuda(),
                             out_dtype=torch.float32, acc_debug=acc)
        expect = sign * xq.to(torch.int64).sum(dim=1)
        assert (acc.cpu().to(torch.int64) == expect[:, None]).all()


def test_forward_extreme_codes_max_k():
    # |acc| reaches 127 * K at the largest K: exactness of the int32 path
    M, N, K = 2, 32, 65536
    xq = torch.full((M, K), 127, dtype=torch.int8)
    xq[1] = -127
    packed = torch.full((N, K // 4), 0x55, dtype=torch.uint8)
    packed[1::2] = 0xAA
    acc = torch.empty((M, N), dtype=torch.int32, device="cuda")
    bl.bitlinear_forward(xq.cuda(), torch.ones(M).cuda(), tiled_cuda(packed, K), torch.ones(N).cuda(),
                         out_dtype=torch.float32, acc_debug=acc)
    a = acc.cpu()
    assert a[0, 0] == 127 * K and a[0, 1] == -127 * K and a[1, 0] == -127 * K


def test_forward_empty_is_noop():
    packed = torch.zeros(bl.bitlinear_packed_bytes(16, 128), dtype=torch.uint8, device="cuda")
    y = bl.bitlinear_forward(torch.zeros((0, 128), dtype=torch.int8, device="cuda"),
                             torch.zeros(0, device="cuda"), packed, torch.ones(16, device="cuda"))
    assert y.shape == (0, 16)


# ---------------------------------------------------------------------------
# full-size workloads: sampled outputs, full x_q / packed comparison
# ---------------------------------------------------------------------------

FULL = []
for wl_name in ("decode_2b", "decode_8b", "prefill_8b_m2048"):
    wl = synth.WORKLOADS[wl_name]
    for M in wl.tokens:
        for pi, p in enumerate(wl.projections):
            FULL.append((wl_name, M, pi))


@pytest.mark.parametrize("wl_name,M,pi", FULL)
def test_full_size_sampled(wl_name, M, pi):
    wl = synth.WORKLOADS[wl_name]
    p = wl.projections[pi]
    dt = torch.float32 if wl.out_dtype == "f32" else torch.bfloat16
    r = run_forward(M, p.N, p.K, dt, seed=synth.weight_seed(wl.seed, 0, pi), outliers=wl.outliers)
    rng = np.random.default_rng(pi + M)
    ts = rng.integers(0, M, 512)
    ns = rng.integers(0, p.N, 512)
    ts[:2] = [0, M - 1]
    ns[:2] = [0, p.N - 1]
    check_output(r, ts, ns)
