"""Pins of the CPU oracle against facts fixed by the pages and by mathematics.

None of these tests re-types an oracle formula and compares it with itself:
each checks a hand-worked example, a closed form, an invariant, a special case
or an exact brute-force computation (Python fractions) on tiny inputs.
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
from oracle import (absmean_gamma, abs_sum_units, act_quant, dequant, pack_codes,
                    rational_to_f32, ternarize, ternary_matmul, ternary_matmul_at,
                    unpack_codes, f32_to_bf16_bits, bf16_bits_to_f64)

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "worked_examples.json")))
EPS32 = np.float32(1e-5)
RMS_EPS = float(np.float32(1e-5))


def bf16(vals):
    return f32_to_bf16_bits(np.asarray(vals, dtype=np.float32))


def rand_bf16(rng, shape, scale=1.0):
    return f32_to_bf16_bits((rng.standard_normal(shape) * scale).astype(np.float32))


# ---------------------------------------------------------------------------
# rounding of a rational to binary32
# ---------------------------------------------------------------------------

def _is_rne(num, den, r):
    """Brute-force check that binary32 r is the nearest value to num/den, ties to even."""
    exact = Fraction(num, den)
    r = np.float32(r)
    up = np.nextafter(r, np.float32(np.inf), dtype=np.float32)
    dn = np.nextafter(r, np.float32(-np.inf), dtype=np.float32)
    d0 = abs(exact - Fraction(float(r)))
    for nb in (up, dn):
        if not np.isfinite(nb):
            continue
        d1 = abs(exact - Fraction(float(nb)))
        if d1 < d0:
            return False
        if d1 == d0:   # tie: r must have an even significand
            if int(np.array(r).view(np.uint32)) & 1:
                return False
    return True


def test_rational_to_f32_is_nearest_even():
    rng = np.random.default_rng(1)
    cases = [(1, 3), (2, 3), (1, 10), (7, 1), (2**24 + 1, 1), (2**24 + 3, 1), (1, 2**149),
             (3, 2**150), (1, 2**151), (5, 2**151), (2**130, 3)]
    for _ in range(400):
        num = int(rng.integers(1, 2**62)) * int(rng.integers(1, 2**40))
        den = int(rng.integers(1, 2**62))
        cases.append((num, den << int(rng.integers(0, 180))))
    for num, den in cases:
        r = rational_to_f32(num, den)
        if np.isinf(r):
            assert Fraction(num, den) >= Fraction(2**128) - Fraction(2**103)
            continue
        assert _is_rne(num, den, r), (num, den, r)
    # exact binary32 values come back unchanged
    for v in [0.1, 3.0, 1e-40, 6e-39, 123456.789, 2.0**-149]:
        f = Fraction(float(np.float32(v)))
        assert rational_to_f32(f.numerator, f.denominator) == np.float32(v)


# ---------------------------------------------------------------------------
# absmean gamma
# ---------------------------------------------------------------------------

def test_abs_sum_exact_equals_fraction_sum():
    rng = np.random.default_rng(2)
    for trial in range(30):
        n = int(rng.integers(1, 300))
        mant = rng.standard_normal(n)
        expo = rng.integers(-160, 120, size=n)
        w = (mant * np.exp2(expo.astype(np.float64))).astype(np.float32)
        w[rng.random(n) < 0.1] = 0.0
        if trial == 0:
            w[:3] = [np.float32(1.4e-45), np.float32(-3e-42), np.float32(3.0e38)]
        exact = sum(abs(Fraction(float(v))) for v in w)
        assert Fraction(abs_sum_units(w), 2**149) == exact


def test_abs_sum_rejects_nonfinite():
    with pytest.raises(ValueError):
        abs_sum_units(np.array([1.0, np.inf], dtype=np.float32))


def test_gamma_is_correctly_rounded_mean():
    rng = np.random.default_rng(3)
    for _ in range(40):
        n = int(rng.integers(1, 200))
        w = (rng.standard_normal(n) * 0.02).astype(np.float32)
        g = absmean_gamma(w)
        exact = sum(abs(Fraction(float(v))) for v in w) / n
        assert _is_rne(exact.numerator, exact.denominator, g)


def test_gamma_differs_from_naive_fp32_sum_only_by_rounding():
    # large sums: the exact mean and a float64 mean agree to far below one fp32 ulp
    rng = np.random.default_rng(4)
    w = (rng.standard_normal(1_000_003) * 0.02).astype(np.float32)
    g = absmean_gamma(w)
    m64 = math.fsum(np.abs(w.astype(np.float64))) / w.size
    assert abs(float(g) - m64) <= 0.5 * float(np.spacing(np.float32(m64))) * (1 + 1e-9)


def test_weights_worked_example():
    ex = GOLDEN["weights_dyadic_2x4"]
    W = np.array(ex["W"], dtype=np.float32)
    packed, gamma, q = oracle.pack_weights(W, np.float32(ex["eps"]))
    assert gamma == np.float32(ex["gamma"])
    assert (q == np.array(ex["w_q"], dtype=np.int8)).all()
    assert (packed == np.array(ex["packed"], dtype=np.uint8)).all()


def test_gamma_and_zero_fraction_statistics_for_gaussian_latents():
    # For W ~ N(0, s^2): E|W| = s*sqrt(2/pi); P(W_q = 0) = P(|W| <= gamma/2)
    # = erf(sqrt(2/pi) / (2*sqrt(2))) = 0.3101 (closed forms).
    rng = np.random.default_rng(5)
    s = 0.02
    W = (rng.standard_normal((1000, 4000)) * s).astype(np.float32)
    g = float(absmean_gamma(W))
    assert abs(g / s - math.sqrt(2 / math.pi)) < 2e-3
    q = ternarize(W, np.float32(g))
    zero_frac = float((q == 0).mean())
    expect = math.erf(math.sqrt(2 / math.pi) / (2 * math.sqrt(2)))
    assert abs(expect - 0.3101) < 1e-4
    assert abs(zero_frac - expect) < 2e-3
    assert abs(float((q == 1).mean()) - float((q == -1).mean())) < 2e-3


# ---------------------------------------------------------------------------
# ternarization
# ---------------------------------------------------------------------------

def test_ternarize_threshold_and_ties():
    gamma = np.float32(0.0123)
    d = np.float32(gamma + EPS32)            # binary32 sum, like the definition's divisor
    half = np.float32(d / np.float32(2))     # exact (power-of-two scaling)
    just_above = np.nextafter(half, np.float32(1), dtype=np.float32)
    just_below = np.nextafter(half, np.float32(0), dtype=np.float32)
    w = np.array([half, -half, just_above, -just_above, just_below,
                  np.float32(1.5) * d, np.float32(2.5) * d, np.float32(100.0), np.float32(-1e-30),
                  np.float32(0.0), np.float32(-0.0)], dtype=np.float32)
    q = ternarize(w, gamma)
    # Round(0.5) = 0 (ties to even); beyond the tie -> +-1; 1.5 -> 2 -> clip 1; 2.5 -> 2 -> clip 1
    assert q.tolist() == [0, 0, 1, -1, 0, 1, 1, 1, 0, 0, 0]


def test_ternarize_idempotent():
    rng = np.random.default_rng(6)
    W = (rng.standard_normal((64, 128)) * 0.02).astype(np.float32)
    _, _, q = oracle.pack_weights(W)
    qf = q.astype(np.float32)
    _, _, q2 = oracle.pack_weights(qf)
    assert (q2 == q).all()


def test_constant_magnitude_and_zero_weights():
    rng = np.random.default_rng(7)
    signs = rng.choice([-1.0, 1.0], size=(16, 32)).astype(np.float32)
    c = np.float32(0.37)
    _, g, q = oracle.pack_weights(signs * c)
    assert g == c
    assert (q == signs.astype(np.int8)).all()
    _, g0, q0 = oracle.pack_weights(np.zeros((8, 16), dtype=np.float32))
    assert g0 == 0 and (q0 == 0).all()


# ---------------------------------------------------------------------------
# 2-bit packing
# ---------------------------------------------------------------------------

def test_pack_code_table_single_weights():
    # [P5-lut]: 00 = 0, 01 = +1, 10 = -1, four per byte
    for j in range(4):
        for v, code in ((1, 1), (-1, 2), (0, 0)):
            q = np.zeros((1, 4), dtype=np.int8)
            q[0, j] = v
            assert pack_codes(q)[0, 0] == code << (2 * j)


def test_pack_roundtrip_and_no_11_codes():
    rng = np.random.default_rng(8)
    q = rng.integers(-1, 2, size=(33, 256)).astype(np.int8)
    p = pack_codes(q)
    assert p.shape == (33, 64)
    assert (unpack_codes(p, 256) == q).all()
    for s in range(4):
        assert (((p >> (2 * s)) & 3) != 3).all()
    with pytest.raises(ValueError):
        pack_codes(np.array([[2, 0, 0, 0]], dtype=np.int8))
    with pytest.raises(ValueError):
        unpack_codes(np.array([[0xC0]], dtype=np.uint8), 4)


# ---------------------------------------------------------------------------
# activation quantization
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("key", ["act_ties_to_even", "act_tie_up"])
def test_act_quant_worked_examples(key):
    ex = GOLDEN[key]
    xq, sigma = act_quant(bf16([ex["x"]]), None, -1.0)
    assert xq[0].tolist() == ex["x_q"]
    assert sigma[0] == max(abs(v) for v in ex["x"]) / 127.0


def test_act_quant_gain_rmsnorm_worked_example():
    ex = GOLDEN["act_gain_rmsnorm"]
    xq, sigma = act_quant(bf16([ex["x"]]), bf16(ex["gain"]), float(np.float32(ex["rms_eps"])))
    assert xq[0].tolist() == ex["x_q"]
    expect = ex["max_xg"] / (127.0 * math.sqrt(ex["mean_sq"] + float(np.float32(ex["rms_eps"]))))
    assert abs(sigma[0] - expect) <= 1e-15 * expect


def _exact_codes(xb, gb):
    """Brute force with exact rationals: Round_half_even(127 * p / max|p|), p = x*g.

    This is the definition for rows whose normalized max|n| = max|p| * r is not
    clamped (r <= 1/sqrt(eps) < 317, so max|p| >= 2^-20 keeps max|n| far above 1e-8
    whenever the row has no tiny values beside it); the callers stay in that range."""
    x = [Fraction(float(v)) for v in bf16_bits_to_f64(xb)]
    g = [Fraction(float(v)) for v in bf16_bits_to_f64(gb)] if gb is not None else [1] * len(x)
    p = [a * b for a, b in zip(x, g)]
    m = max(abs(v) for v in p)
    assert m >= Fraction(1, 2**20)
    return [max(-128, min(127, round(127 * v / m))) for v in p]


@pytest.mark.parametrize("key", ["act_clamp_regular_tiny_row", "act_clamp_plain_tiny_row",
                                 "act_clamp_small_rmsnorm_row"])
def test_act_quant_clamp_worked_examples(key):
    # activation_quant clamps the max of the RMSNorm output, not of the raw row
    ex = GOLDEN[key]
    xb = bf16([ex["x"]])
    assert (bf16_bits_to_f64(xb)[0] == np.array(ex["x"])).all()
    xq, sigma = act_quant(xb, None, float(np.float32(ex["rms_eps"])) if ex["rms_eps"] >= 0 else -1.0)
    assert xq[0].tolist() == ex["x_q"]
    if "sigma_den" in ex:
        assert sigma[0] == float(np.float32(1e-8)) / ex["sigma_den"]


def test_act_quant_zero_row_takes_the_clamp():
    # an all-zero row: zero codes and the clamped scale 1e-8 / 127, with or without RMSNorm
    z = np.zeros((2, 64), dtype=np.uint16)
    for eps in (RMS_EPS, -1.0):
        zq, zs = act_quant(z, None, eps)
        assert (zq == 0).all() and (zs == float(np.float32(1e-8)) / 127.0).all()


def test_f32_to_bf16_bits_golden():
    ex = GOLDEN["bf16_round_nearest_even"]
    src = np.array([int(a, 16) for a, _, _ in ex["cases"]], dtype=np.uint32).view(np.float32)
    want = [int(b, 16) for _, b, _ in ex["cases"]]
    got = f32_to_bf16_bits(src).tolist()
    assert got == want, [(c[2], hex(g)) for c, g in zip(ex["cases"], got) if int(c[1], 16) != g]


def test_act_quant_matches_exact_rational_bruteforce():
    rng = np.random.default_rng(9)
    for trial in range(60):
        K = int(rng.integers(1, 40))
        xb = rand_bf16(rng, (1, K), scale=float(np.exp2(rng.integers(-20, 20))))
        gb = rand_bf16(rng, (K,)) if trial % 2 else None
        xq, _ = act_quant(xb, gb, RMS_EPS)
        assert xq[0].tolist() == _exact_codes(xb[0], gb)


def test_act_quant_constructed_ties_bruteforce():
    # rows whose 127*p/m hit half-integers: m = 127 * 2^j makes the quotient p / 2^j
    rng = np.random.default_rng(10)
    for j in range(-3, 4):
        vals = np.concatenate([[127.0 * 2.0**j], (rng.integers(-254, 255, size=31) / 2.0) * 2.0**j])
        xb = bf16([vals])
        xq, _ = act_quant(xb, None, RMS_EPS)
        assert xq[0].tolist() == _exact_codes(xb[0], None)


def test_act_quant_invariants():
    rng = np.random.default_rng(11)
    M, K = 7, 300
    xb = rand_bf16(rng, (M, K), 3.0)
    gb = f32_to_bf16_bits(rng.uniform(0.5, 1.5, K).astype(np.float32))
    xq, sig = act_quant(xb, gb, RMS_EPS)
    x = bf16_bits_to_f64(xb)
    g = bf16_bits_to_f64(gb)
    p = x * g
    # range, and the argmax element maps to +-127
    assert xq.min() >= -127 and xq.max() <= 127
    for t in range(M):
        k = int(np.argmax(np.abs(p[t])))
        assert xq[t, k] == 127 * np.sign(p[t, k])
    # sign symmetry: quant(-x) = -quant(x)
    xq_neg, sig_neg = act_quant(xb ^ np.uint16(0x8000), gb, RMS_EPS)
    assert (xq_neg == -xq).all() and (sig_neg == sig).all()
    # power-of-two scale invariance of the codes (bf16 exact)
    for j in (-5, 3):
        xs = f32_to_bf16_bits((x * 2.0**j).astype(np.float32))
        assert (bf16_bits_to_f64(xs) == x * 2.0**j).all()
        assert (act_quant(xs, gb, RMS_EPS)[0] == xq).all()
    # permutation equivariance over k
    perm = rng.permutation(K)
    assert (act_quant(xb[:, perm], gb[perm], RMS_EPS)[0] == xq[:, perm]).all()
    # idempotence: quantizing the codes themselves returns them
    xq2, _ = act_quant(f32_to_bf16_bits(xq.astype(np.float32)), None, -1.0)
    assert (xq2 == xq).all()
    # a gain that is a constant power of two changes nothing in the codes
    g2 = f32_to_bf16_bits(np.full(K, 4.0, dtype=np.float32))
    assert (act_quant(xb, g2, RMS_EPS)[0] == act_quant(xb, None, RMS_EPS)[0]).all()
    # zero row: zero codes, finite scale
    z = np.zeros((1, K), dtype=np.uint16)
    zq, zs = act_quant(z, gb, RMS_EPS)
    assert (zq == 0).all() and np.isfinite(zs).all()


def test_act_scale_reconstructs_rmsnorm_output():
    # sigma * x_q must reproduce the RMSNorm output n = x * g / sqrt(mean(x^2)+eps)
    # within half a quantization step (nn.RMSNorm definition, computed here in fp64)
    rng = np.random.default_rng(12)
    M, K = 9, 512
    xb = rand_bf16(rng, (M, K), 1.0)
    gb = f32_to_bf16_bits(rng.uniform(0.5, 1.5, K).astype(np.float32))
    xq, sig = act_quant(xb, gb, RMS_EPS)
    x = bf16_bits_to_f64(xb)
    g = bf16_bits_to_f64(gb)
    n = x * g / np.sqrt((x * x).mean(axis=1, keepdims=True) + RMS_EPS)
    err = np.abs(n - sig[:, None] * xq)
    assert (err <= 0.5 * sig[:, None] * (1 + 1e-9)).all()
    # and sigma is max|n| / 127
    assert np.allclose(sig, np.abs(n).max(axis=1) / 127.0, rtol=1e-13, atol=0)


def test_outlier_rows_push_codes_small():
    # statistics check: a x20 outlier compresses the rest of the row into small codes
    rng = np.random.default_rng(13)
    x = rng.standard_normal((64, 1024)).astype(np.float32)
    mask = rng.random(x.shape) < 0.01
    xo = np.where(mask, x * 20, x).astype(np.float32)
    q_plain, _ = act_quant(f32_to_bf16_bits(x), None, RMS_EPS)
    q_out, _ = act_quant(f32_to_bf16_bits(xo), None, RMS_EPS)
    assert np.median(np.abs(q_out[~mask])) < 0.3 * np.median(np.abs(q_plain))


# ---------------------------------------------------------------------------
# contraction and dequantization
# ---------------------------------------------------------------------------

def test_contraction_weight_invariants():
    rng = np.random.default_rng(14)
    xq = rng.integers(-127, 128, size=(5, 96)).astype(np.int8)
    ones = np.ones((7, 96), dtype=np.int8)
    rowsum = xq.astype(np.int64).sum(axis=1)
    assert (ternary_matmul(xq, ones) == rowsum[:, None]).all()
    assert (ternary_matmul(xq, -ones) == -rowsum[:, None]).all()
    assert (ternary_matmul(xq, 0 * ones) == 0).all()


def test_contraction_equals_mask_form():
    # [P5-mask]: y = (W==1) x - (W==-1) x
    rng = np.random.default_rng(15)
    xq = rng.integers(-127, 128, size=(6, 200)).astype(np.int8)
    wq = rng.integers(-1, 2, size=(50, 200)).astype(np.int8)
    xf = xq.astype(np.float64)
    mask = (wq == 1).astype(np.float64) @ xf.T - (wq == -1).astype(np.float64) @ xf.T
    assert (ternary_matmul(xq, wq) == mask.T.astype(np.int64)).all()


def test_contraction_exhaustive_k4():
    # every one of the 3^4 weight rows against extreme and small activations
    rows = np.array(np.meshgrid(*[[-1, 0, 1]] * 4, indexing="ij")).reshape(4, -1).T.astype(np.int8)
    vals = [-127, -1, 0, 1, 127]
    xs = np.array(np.meshgrid(*[vals] * 4, indexing="ij")).reshape(4, -1).T.astype(np.int8)
    acc = ternary_matmul(xs, rows)
    for i in range(0, len(xs), 37):
        for j in range(len(rows)):
            assert acc[i, j] == sum(int(a) * int(b) for a, b in zip(xs[i], rows[j]))


def test_forward_matches_dense_float_bruteforce():
    # y equals a plain fp64 dense matmul of the dequantized operands on tiny shapes
    rng = np.random.default_rng(16)
    for M, N, K in [(1, 3, 4), (3, 5, 8), (8, 8, 8), (2, 7, 16)]:
        W = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
        xb = rand_bf16(rng, (M, K))
        out = oracle.bitlinear_forward(xb, None, RMS_EPS, W)
        xdq = out["x_q"].astype(np.float64) * out["sigma"][:, None]
        wdq = out["w_q"].astype(np.float64) * float(out["gamma"])
        dense = xdq @ wdq.T
        bound = 1e-12 * (np.abs(xdq) @ np.abs(wdq).T)   # fp64 rounding of the dense sum
        assert (np.abs(out["y"] - dense) <= bound).all()


def test_matmul_at_matches_full():
    rng = np.random.default_rng(17)
    xq = rng.integers(-127, 128, size=(9, 64)).astype(np.int8)
    wq = rng.integers(-1, 2, size=(11, 64)).astype(np.int8)
    full = ternary_matmul(xq, wq)
    ts = rng.integers(0, 9, 40)
    ns = rng.integers(0, 11, 40)
    assert (ternary_matmul_at(xq, wq, ts, ns) == full[ts, ns]).all()


def test_dequant_worked_example():
    ex = GOLDEN["dequant_single"]
    y = dequant(np.array([[ex["acc"]]], dtype=np.int32), np.array([ex["sigma"]]), np.array([ex["w_scale"]]))
    assert y[0, 0] == ex["y"]


# ---------------------------------------------------------------------------
# the linear stack (block_layer)
# ---------------------------------------------------------------------------

def _rand_layer(rng, H, NQKV, F, zero=()):
    layer = {}
    for name, (n, k) in {"qkv": (NQKV, H), "o": (H, H), "gate_up": (2 * F, H), "down": (H, F)}.items():
        wq = np.zeros((n, k), np.int8) if name in zero else rng.integers(-1, 2, (n, k)).astype(np.int8)
        layer[name] = wq
        layer[name + "_scale"] = np.full(n, 0.01 + 0.001 * len(name))
    for name, k in {"gain_qkv": H, "gain_o": H, "gain_gate_up": H, "gain_down": F}.items():
        layer[name] = oracle.f32_to_bf16_bits(rng.uniform(0.5, 1.5, k).astype(np.float32))
    return layer


def test_relu2_gate_closed_form():
    g = np.array([-2.0, 0.0, 1.5, 3.0, 2.0], np.float32)
    u = np.array([5.0, 7.0, 2.0, -1.0, 0.125], np.float32)
    h = oracle.bf16_bits_to_f64(oracle.relu2_gate_bits(g, u))
    assert list(h) == [0.0, 0.0, 4.5, -9.0, 0.5]
    # rounding: 1.1^2 * 1 in fp32, then to bf16 nearest
    h2 = oracle.bf16_bits_to_f64(oracle.relu2_gate_bits(np.array([1.1], np.float32), np.array([1.0], np.float32)))
    assert h2[0] == oracle.bf16_bits_to_f64(oracle.f32_to_bf16_bits(np.float32(1.1) * np.float32(1.1)))[0]


def test_block_layer_zero_projections_keep_the_residual_stream():
    rng = np.random.default_rng(5)
    H, NQKV, F, M = 32, 48, 64, 3
    x = oracle.f32_to_bf16_bits(rng.standard_normal((M, H)).astype(np.float32))
    for zero in (("o", "down"), ("qkv", "o", "gate_up", "down")):
        out = oracle.block_layer(x, _rand_layer(rng, H, NQKV, F, zero=zero), 1e-5)
        assert (out == x).all()


def test_block_layer_matches_dense_fp64_recomputation():
    # the same stages with dense fp64 matmuls of dequantized operands
    rng = np.random.default_rng(6)
    H, NQKV, F, M = 16, 24, 32, 4
    layer = _rand_layer(rng, H, NQKV, F)
    x = oracle.f32_to_bf16_bits((3 * rng.standard_normal((M, H))).astype(np.float32))

    def lin(xb, gain, w, ws):
        xq, sig = oracle.act_quant(xb, gain, 1e-5)
        return ((xq.astype(np.float64) * sig[:, None]) @ (w.astype(np.float64) * ws[:, None]).T).astype(np.float32)

    x32 = oracle.bf16_bits_to_f64(x).astype(np.float32)
    qkv = lin(x, layer["gain_qkv"], layer["qkv"], layer["qkv_scale"])
    q = oracle.f32_to_bf16_bits(np.ascontiguousarray(qkv[:, :H]))
    xb = oracle.f32_to_bf16_bits(x32 + lin(q, layer["gain_o"], layer["o"], layer["o_scale"]))
    gu = lin(xb, layer["gain_gate_up"], layer["gate_up"], layer["gate_up_scale"])
    r = np.maximum(gu[:, :F], np.float32(0))
    h = oracle.f32_to_bf16_bits((r * r) * gu[:, F:])
    x2 = oracle.bf16_bits_to_f64(xb).astype(np.float32)
    expect = oracle.f32_to_bf16_bits(x2 + lin(h, layer["gain_down"], layer["down"], layer["down_scale"]))
    assert (oracle.block_layer(x, layer, 1e-5) == expect).all()


# ---------------------------------------------------------------------------
# scale-granularity variants: per-output-channel weight scale, per-tensor Q_b = 128
# ---------------------------------------------------------------------------

def test_pack_per_channel_worked_example():
    ex = GOLDEN["weights_per_channel_2x4"]
    W = np.array(ex["W"], dtype=np.float32)
    packed, gammas, wq = oracle.pack_weights_per_channel(W, np.float32(ex["eps"]))
    assert gammas.tolist() == ex["gamma"]
    assert wq.tolist() == ex["w_q"]
    assert packed.tolist() == ex["packed"]
    # the per-tensor packing of the same matrix zeroes the small row
    _, g, q = oracle.pack_weights(W, np.float32(ex["eps"]))
    assert float(g) == ex["per_tensor_gamma"] and q.tolist() == ex["per_tensor_w_q"]


def test_pack_per_channel_rows_are_one_row_matrices():
    # each row's scale and codes are those of that row packed alone (a 1 x K matrix),
    # whose per-tensor absmean is pinned above
    rng = np.random.default_rng(21)
    W = (rng.standard_normal((9, 40)) * np.exp2(rng.integers(-6, 4, (9, 1)))).astype(np.float32)
    _, gammas, wq = oracle.pack_weights_per_channel(W)
    for n in range(9):
        _, g, q = oracle.pack_weights(W[n:n + 1])
        assert gammas[n] == g and (wq[n] == q[0]).all()


def test_pack_per_channel_equals_per_tensor_for_rows_of_equal_magnitudes():
    # rows that are sign flips and permutations of one row share its mean |W|: one scale
    rng = np.random.default_rng(22)
    base = (rng.standard_normal(64) * 0.02).astype(np.float32)
    W = np.stack([rng.permutation(base) * rng.choice([-1.0, 1.0], 64).astype(np.float32) for _ in range(6)])
    _, gammas, wq = oracle.pack_weights_per_channel(W)
    _, g, q = oracle.pack_weights(W)
    assert (gammas == g).all() and (wq == q).all()


def test_pack_per_channel_row_scaling_by_powers_of_two():
    # with eps = 0, scaling row n by 2^j scales its gamma by 2^j exactly and keeps its codes
    rng = np.random.default_rng(23)
    W = (rng.standard_normal((5, 96)) * 0.02).astype(np.float32)
    s = np.exp2(np.array([-3, 0, 2, 5, -1], dtype=np.float32))[:, None]
    _, g1, q1 = oracle.pack_weights_per_channel(W, np.float32(0.0))
    _, g2, q2 = oracle.pack_weights_per_channel((W * s).astype(np.float32), np.float32(0.0))
    assert (g2 == g1 * s[:, 0]).all() and (q1 == q2).all()


@pytest.mark.parametrize("key", ["act_per_tensor_q128", "act_per_tensor_tiny"])
def test_act_quant_per_tensor_worked_examples(key):
    ex = GOLDEN[key]
    xb = bf16(ex["x"])
    assert (bf16_bits_to_f64(xb) == np.array(ex["x"])).all()
    xq, sigma = oracle.act_quant_per_tensor(xb)
    assert xq.tolist() == ex["x_q"]
    want = ex["sigma"] if "sigma" in ex else 2.0 ** ex["sigma_log2"]
    assert (sigma == want).all()


def test_act_quant_per_tensor_dyadic_bruteforce():
    # with max|x| = 2^j (j >= -2: 1e-8 is below half an ulp of 2^j) the 1e-8 vanishes in
    # binary32 and x 128 / 2^j is exact: the codes are Round(Clip(x 128 / 2^j, -128, 127))
    # in exact rationals
    rng = np.random.default_rng(24)
    for trial in range(40):
        M, K = int(rng.integers(1, 5)), int(rng.integers(1, 48))
        j = int(rng.integers(-2, 8))
        x = (rng.uniform(-1, 1, (M, K)) * 2.0**j).astype(np.float32)
        x.flat[int(rng.integers(0, M * K))] = (2.0**j) * (1 if trial % 2 else -1)
        xb = f32_to_bf16_bits(x)
        xv = bf16_bits_to_f64(xb)
        xq, sigma = oracle.act_quant_per_tensor(xb)
        g = Fraction(2) ** j
        for t in range(M):
            for k in range(K):
                v = Fraction(float(xv[t, k])) * 128 / g
                v = min(max(v, Fraction(-128)), Fraction(127))
                assert xq[t, k] == round(v)
        assert (sigma == float(g) / 128).all()
    # one scale for the whole tensor: a row's codes depend on the other rows
    x = np.array([[1.0, 0.5], [4.0, -0.25]], dtype=np.float32)
    xq, _ = oracle.act_quant_per_tensor(f32_to_bf16_bits(x))
    assert xq[0].tolist() == [32, 16]
