"""CPU checks of the index maps and byte tables that the decode kernels
(csrc/decode_dp4a.cu, csrc/decode_tc.cu) rely on, restated here in numpy: they need no GPU.

* Reading the tile-major packed layout chunk by chunk (lane c of a row takes the
  16-byte chunk c of every 512-wide segment, at position c ^ (r % 8)), expanding
  each 32-bit word of codes with the byte-permute table 0x00FF0100 into the
  int8 words of inputs (0,2,4,6), (8..14 even), (1,3,5,7), (9..15 odd), and
  permuting the activations the same way (selectors 0x6420 / 0x7531) gives the
  exact ternary product of the oracle.
* The thread-to-row maps cover every padded row once; the staged activation
  chunks (80-byte pitch) are read by the eight chunk lanes of a warp without
  shared-memory bank conflicts.
* The tensor-core kernels' e4m3 weight table and the split of every int8 code
  into two exact e4m3 values (from the format's definition).
"""
import numpy as np
import pytest

import oracle
from bitlinear_rmsnorm_token_int8_b300 import layout

CODE_TO_I8 = 0x00FF0100
SEG_PITCH, CHUNK_PITCH = 640, 80


def byte_perm(a: int, b: int, sel: int) -> int:
    """PRMT in its default mode: result byte i = byte (nibble i of sel) & 7 of {b:a}."""
    src = (b << 32) | a
    out = 0
    for i in range(4):
        k = (sel >> (4 * i)) & 7
        out |= ((src >> (8 * k)) & 0xFF) << (8 * i)
    return out


def i8x4(w: int) -> np.ndarray:
    return np.array([(w >> (8 * i)) & 0xFF for i in range(4)], dtype=np.uint8).view(np.int8).astype(np.int64)


def expand_word(w: int):
    lo, hi = w & 0x33333333, (w >> 2) & 0x33333333
    return [byte_perm(CODE_TO_I8, 0, lo), byte_perm(CODE_TO_I8, 0, lo >> 16),
            byte_perm(CODE_TO_I8, 0, hi), byte_perm(CODE_TO_I8, 0, hi >> 16)]


def permute16(x16: np.ndarray):
    v = [int.from_bytes(x16[4 * i:4 * i + 4].astype(np.int8).tobytes(), "little") for i in range(4)]
    return [byte_perm(v[0], v[1], 0x6420), byte_perm(v[2], v[3], 0x6420), byte_perm(v[0], v[1], 0x7531),
            byte_perm(v[2], v[3], 0x7531)]


@pytest.mark.parametrize("N,K,KS", [(16, 512, 1), (144, 1536, 2), (130, 2560, 1), (48, 6912, 4), (272, 640, 2)])
def test_code_kernel_reading_gives_the_ternary_product(N, K, KS):
    rng = np.random.default_rng(N + K)
    wq = rng.integers(-1, 2, (N, K)).astype(np.int8)
    x = rng.integers(-127, 128, K).astype(np.int8)
    tiled = layout.tiled_from_canonical(oracle.pack_codes(wq), K)
    nseg = -(-K // 512)
    Np = -(-N // 16) * 16
    xp = np.zeros(nseg * 512, dtype=np.int8)
    xp[:K] = x
    want = oracle.ternary_matmul(x[None, :], wq)[0]
    for n in range(N):
        t, r = n // 128, n % 128
        R = min(128, Np - 128 * t)
        total = 0
        for ks in range(KS):                          # the row's 8 KS lanes
            for c in range(8):
                for s in range(ks, nseg, KS):
                    off = t * nseg * 16384 + s * R * 128 + r * 128 + ((c ^ (r & 7)) << 4)
                    chunk = tiled[off:off + 16]
                    for j in range(4):
                        w = int.from_bytes(chunk[4 * j:4 * j + 4].tobytes(), "little")
                        k0 = s * 512 + c * 64 + 16 * j
                        for ww, xx in zip(expand_word(w), permute16(xp[k0:k0 + 16])):
                            total += int((i8x4(ww) * i8x4(xx)).sum())      # one dp4a
        assert total == want[n]


def test_code_table_and_selectors():
    # codes 0, 1, 2 -> 0, +1, -1 as int8 bytes; the words hold inputs in the order above
    assert [byte_perm(CODE_TO_I8, 0, c) & 0xFF for c in range(3)] == [0x00, 0x01, 0xFF]
    x = np.arange(16, dtype=np.int8)
    got = [i8x4(w).tolist() for w in permute16(x)]
    assert got == [[0, 2, 4, 6], [8, 10, 12, 14], [1, 3, 5, 7], [9, 11, 13, 15]]


@pytest.mark.parametrize("Np", [16, 144, 2560, 13824])
@pytest.mark.parametrize("KS", [1, 2, 4])
def test_row_maps_cover_each_row_once(Np, KS):
    # contraction kernel: 4 warps, 4 / KS rows per warp, grid Np KS / 16
    rows = []
    for b in range(Np * KS // 16):
        for warp in range(4):
            for lane in range(0, 32, 8 * KS):
                rows.append((b * 4 + warp) * (4 // KS) + (lane >> (3 + KS.bit_length() - 1)))
    assert sorted(rows) == list(range(Np))
    # one-token layer kernel: T threads, (T / 32) 4 / KS rows per CTA, ceil(Np / that) CTAs
    for T in (128, 256, 512):
        per = (T // 32) * 4 // KS
        seen = []
        for b in range(-(-Np // per)):
            for warp in range(T // 32):
                for lane in range(0, 32, 8 * KS):
                    row = (b * (T // 32) + warp) * (4 // KS) + (lane >> (3 + KS.bit_length() - 1))
                    if row < Np:
                        seen.append(row)
        assert sorted(seen) == list(range(Np))


def test_staging_offsets_and_banks():
    # group g of 16 inputs -> segment g / 32, chunk (g / 4) % 8, word g % 4: distinct,
    # in range, and the eight chunk lanes of a warp reading word j hit distinct banks
    nseg = 14
    offs = {(g >> 5) * SEG_PITCH + ((g >> 2) & 7) * CHUNK_PITCH + 16 * (g & 3) for g in range(nseg * 32)}
    assert len(offs) == nseg * 32 and max(offs) + 16 <= nseg * SEG_PITCH
    for j in range(4):
        banks = [((c * CHUNK_PITCH + 16 * j) // 4 + b) % 32 for c in range(8) for b in range(4)]
        assert len(set(banks)) == 32


def e4m3_value(b: int) -> float:
    """OCP FP8 E4M3: sign, 4 exponent bits (bias 7), 3 mantissa bits; exponent 0 is subnormal."""
    s = -1.0 if b & 0x80 else 1.0
    e, m = (b >> 3) & 0xF, b & 7
    return s * (m / 8.0) * 2.0 ** -6 if e == 0 else s * (1.0 + m / 8.0) * 2.0 ** (e - 7)


def test_tensor_core_operand_split_is_exact():
    # the tcgen05 kernels' weight table 0x00B83800: codes 0, 1, 2 -> e4m3 0, +1, -1
    table = 0x00B83800
    assert [e4m3_value((table >> (8 * c)) & 0xFF) for c in range(3)] == [0.0, 1.0, -1.0]
    # every int8 code x = 16 h + l with h = floor((x + 8) / 16) in [-8, 8] and l in [-8, 7],
    # both exact e4m3 values, so two e4m3 products per code reproduce x exactly
    exact = {e4m3_value(b) for b in range(256) if (b & 0x7F) != 0x7F}
    for x in range(-127, 128):
        h = (x + 8) // 16
        l = x - 16 * h
        assert -8 <= h <= 8 and -8 <= l <= 7
        assert float(h) in exact and float(l) in exact and 16 * h + l == x
    # the fp32 accumulators stay exact integers: one plane's column sums |h| or |l| <= 8
    # times K <= 65536 ternary weights, at most 2^19; the decode kernel adds 16 h-sums and
    # the l-sums in int32, and the prefill kernel's single accumulator is bounded by 127 K
    assert 8 * 65536 <= 2 ** 24 and 127 * 65536 <= 2 ** 24


# ---- the one-token layer kernel's statistics equal the quantization kernel's --------
# Both reduce (max|x g|, sum x^2 as an fp32 pair) with the same per-thread order and
# xor trees; the layer kernel only has more warps, whose partials are zero.  Restated
# in float32 numpy (IEEE round to nearest even, like the GPU's __fadd_rn and friends).

F32 = np.float32


def _two_sum(a, b):
    s = F32(a + b)
    bb = F32(s - a)
    return s, F32(F32(a - F32(s - bb)) + F32(b - bb))


def _pair_add(h1, l1, h2, l2):
    s, e = _two_sum(h1, h2)
    e = F32(e + F32(l1 + l2))
    h = F32(s + e)
    return h, F32(e - F32(h - s))


def _xor_tree(vals):
    """vals: 32 lanes of (amax, hi, lo); returns lane 0 after offsets 16, 8, 4, 2, 1."""
    v = list(vals)
    for o in (16, 8, 4, 2, 1):
        nv = []
        for i in range(32):
            a1, h1, l1 = v[i]
            a2, h2, l2 = v[i ^ o]
            h, l = _pair_add(h1, l1, h2, l2)
            nv.append((max(a1, a2), h, l))
        v = nv
    return v[0]


def _row_stats(x, g, T):
    U = len(x) // 16
    per = []
    for t in range(T):
        a, hi, lo = F32(0), F32(0), F32(0)
        if t < U:
            for j in range(16):
                xv, gv = x[16 * t + j], g[16 * t + j]
                a = max(a, abs(F32(xv * gv)))
                s, e = _two_sum(hi, F32(xv * xv))
                hi, lo = s, F32(lo + e)
        per.append((a, hi, lo))
    warps = [_xor_tree(per[32 * w:32 * w + 32]) for w in range(T // 32)]
    lanes = [warps[i] if i < len(warps) else (F32(0), F32(0), F32(0)) for i in range(32)]
    a, h, l = _xor_tree(lanes)
    return a, F32(h + l)


@pytest.mark.parametrize("K", [128, 1152, 2560, 6912])
def test_layer_kernel_statistics_equal_the_quantization_kernels(K):
    rng = np.random.default_rng(K)
    # bf16-valued inputs and gains (8 significant bits), wide exponent range
    x = (rng.standard_normal(K) * np.exp2(rng.integers(-6, 7, K))).astype(np.float32)
    x = (x.view(np.uint32) & 0xFFFF0000).view(np.float32)
    g = (rng.uniform(0.5, 1.5, K).astype(np.float32).view(np.uint32) & 0xFFFF0000).view(np.float32)
    tq = (K // 16 + 31) // 32 * 32            # the quantization kernel's threads for one row
    tf = (tq + 127) // 128 * 128              # the layer kernel's
    a1, s1 = _row_stats(x, g, tq)
    a2, s2 = _row_stats(x, g, tf)
    assert a1 == a2 and s1.view(np.uint32) == s2.view(np.uint32)
    # and the pair sum is the exact sum of squares rounded once, for these inputs
    exact = sum(int(v) for v in (x.astype(np.float64) ** 2 * 2.0 ** 300).astype(object))
    assert abs(float(s1) - float(np.float64(exact) * 2.0 ** -300)) <= np.spacing(s1)


# ---------------------------------------------------------------------------
# prefill_tc.cu: the persistent grid's cluster tiles (launch_prefill_tc and the
# loops of the producers, decoders and epilogue)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("M,N,CL,TT", [
    (256, 19200, 2, 256), (500, 10240, 2, 256), (2048, 14336, 2, 256), (2048, 4096, 2, 256),
    (600, 512, 2, 128), (38400, 128, 1, 256), (4000, 1280, 1, 128), (1000, 9728, 2, 128), (33, 48, 1, 128)])
def test_prefill_tiles_cover_every_row_and_token_once(M, N, CL, TT):
    sms = 148
    nwb = (N + 127) // 128
    nwbg = (nwb + CL - 1) // CL                            # weight-block groups
    ntok = (M + TT - 1) // TT
    ctiles = nwbg * ntok
    clusters = min(sms // CL, ctiles)
    Mp = (M + 255) // 256 * 256
    seen = np.zeros((nwbg * CL, Mp), dtype=np.int32)
    for cid in range(clusters):                            # each cluster's persistent loop
        for ct in range(cid, ctiles, clusters):
            for rank in range(CL):
                wb, tt = (ct % nwbg) * CL + rank, ct // nwbg
                seen[wb, tt * TT:(tt + 1) * TT] += 1
    assert (seen[:, :M] == 1).all()                        # every weight block and token once
    assert (seen[:nwb, M:] <= 1).all()
    assert clusters * CL <= sms
