/*
 * CPU oracle for the BitNet b1.58 BitLinear forward.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may load this file's
 * library: only the tests, the package's smoke check and the CPU-baseline leg of
 * the benchmark call it.  It shares no code, header, table or constant generator
 * with the CUDA library, and it is deliberately plain: single-threaded loops, no
 * SIMD intrinsics, no OpenMP, no blocking or reordering beyond what the stated
 * definitions need.  Build flags: -O2 -ffp-contract=off (no FMA contraction), no
 * fast-math; binary32 arithmetic is the SSE one of x86-64 (FLT_EVAL_METHOD == 0).
 *
 * Sources (pages and the section on each):
 *   [P4-eq]  "BitNet b1.58 in Production: 1-Bit LLMs and Energy Benchmarks",
 *            section "The Mathematical Mechanism: BitLinear vs Standard Linear",
 *            items 1-4 (absmean weight quantization, absmax activation
 *            quantization, integer addition kernel, dequantization by
 *            gamma*max|x|/Q_b).
 *   [P4-code] same page, "Production Multi-File Implementation", bit_linear.py
 *            (weight_quant, activation_quant, BitLinear.forward with RMSNorm).
 *   [P5-lut] "BitNet 1-bit LLM Inference Framework", section "How the LUT
 *            Kernel Works" (2-bit code 00=0, 01=+1, 10=-1, four weights per
 *            byte; integer accumulation by conditional add / subtract).
 *   [P3-how] "BitNet (1-bit LLMs)", section "How It Works", item 3 (adds and
 *            subtracts of 8-bit activations replace multiplications).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

/* ------------------------------------------------------------------------- */
/* absmean: exact sum of |W|                                                 */
/* ------------------------------------------------------------------------- */

/*
 * [P4-eq] item 1: gamma = (1/(n m)) * sum_ij |W_ij|.
 *
 * Every finite binary32 value is an integer multiple of 2^-149, so the sum of
 * |W| is an integer count of 2^-149 units.  This routine adds those integers
 * exactly into a fixed-point accumulator of base-2^32 digits (little-endian)
 * and returns them in digits[0..ndigits).  The division by n*m and the single
 * rounding to binary32 are done by the Python side with unbounded integers.
 *
 * Returns 0, or -1 if some value is Inf/NaN, or -2 if ndigits < 12.
 */
int oracle_abs_sum_exact(const float *w, int64_t n, uint32_t *digits, int ndigits)
{
    uint64_t acc[16];
    int64_t i;
    int j;
    if (ndigits < 12 || ndigits > 16) return -2;
    memset(acc, 0, sizeof(acc));
    for (i = 0; i < n; ++i) {
        uint32_t bits;
        uint32_t e, mant, pos, limb, off;
        uint64_t v;
        memcpy(&bits, &w[i], 4);
        bits &= 0x7fffffffu;                 /* |w| */
        e = bits >> 23;
        mant = bits & 0x7fffffu;
        if (e == 255u) return -1;
        if (e != 0u) {                       /* normal: 1.m * 2^(e-127) = mant24 * 2^(e-1) units */
            mant |= 0x800000u;
            pos = e - 1u;
        } else {                             /* subnormal: mant * 2^-149 = mant units */
            pos = 0u;
        }
        limb = pos >> 5;
        off = pos & 31u;
        v = (uint64_t)mant << off;           /* at most 55 bits */
        acc[limb] += v & 0xffffffffu;
        acc[limb + 1] += v >> 32;
        if ((i & 0x3fffffff) == 0x3fffffff) { /* keep every digit below 2^63 */
            uint64_t carry = 0;
            for (j = 0; j < 16; ++j) {
                uint64_t t = acc[j] + carry;
                acc[j] = t & 0xffffffffu;
                carry = t >> 32;
            }
        }
    }
    {
        uint64_t carry = 0;
        for (j = 0; j < 16; ++j) {
            uint64_t t = acc[j] + carry;
            acc[j] = t & 0xffffffffu;
            carry = t >> 32;
        }
    }
    for (j = 0; j < ndigits; ++j) digits[j] = (uint32_t)acc[j];
    return 0;
}

/* ------------------------------------------------------------------------- */
/* ternarization                                                             */
/* ------------------------------------------------------------------------- */

/*
 * [P4-eq] item 1 and [P4-code] weight_quant:
 *   W_q = Clip(Round(W / (gamma + eps)), -1, 1)
 * with gamma the binary32 absmean and eps = 1e-5 (binary32), so the divisor
 * is d = fl32(gamma + eps).  W / d is formed in binary64 and rounded to the
 * nearest integer with ties to even (torch.round semantics), then clipped.
 */
void oracle_ternarize(const float *w, int64_t n, float gamma, float eps, int8_t *q)
{
    float d = gamma + eps;                   /* one binary32 rounding */
    int64_t i;
    for (i = 0; i < n; ++i) {
        double r = rint((double)w[i] / (double)d);
        if (r > 1.0) r = 1.0;
        if (r < -1.0) r = -1.0;
        q[i] = (int8_t)r;
    }
}

/*
 * [P5-lut]: four ternary weights per byte with the 2-bit code 00 = 0,
 * 01 = +1, 10 = -1 (11 is never written).  Within a row (an output feature)
 * weight k sits in byte k/4 of the row at bits 2*(k%4) .. 2*(k%4)+1, so row n
 * starts at byte n*K/4.  K must be a multiple of 4.  Returns the number of
 * values that are not in {-1, 0, +1} (nothing is written for those).
 */
int64_t oracle_pack_codes(const int8_t *q, int64_t N, int64_t K, uint8_t *packed)
{
    int64_t n, k, bad = 0;
    for (n = 0; n < N; ++n) {
        for (k = 0; k < K; k += 4) {
            uint8_t byte = 0;
            int s;
            for (s = 0; s < 4; ++s) {
                int8_t v = q[n * K + k + s];
                uint8_t code;
                if (v == 0) code = 0u;
                else if (v == 1) code = 1u;
                else if (v == -1) code = 2u;
                else { ++bad; code = 0u; }
                byte = (uint8_t)(byte | (code << (2 * s)));
            }
            packed[n * (K / 4) + k / 4] = byte;
        }
    }
    return bad;
}

/* Inverse of oracle_pack_codes.  Returns the number of 11 codes met (decoded as 0). */
int64_t oracle_unpack_codes(const uint8_t *packed, int64_t N, int64_t K, int8_t *q)
{
    int64_t n, k, bad = 0;
    for (n = 0; n < N; ++n) {
        for (k = 0; k < K; ++k) {
            uint8_t code = (uint8_t)((packed[n * (K / 4) + k / 4] >> (2 * (k % 4))) & 3u);
            int8_t v;
            if (code == 0u) v = 0;
            else if (code == 1u) v = 1;
            else if (code == 2u) v = -1;
            else { ++bad; v = 0; }
            q[n * K + k] = v;
        }
    }
    return bad;
}

/* ------------------------------------------------------------------------- */
/* RMSNorm + per-token absmax int8 activation quantization                   */
/* ------------------------------------------------------------------------- */

static double bf16_to_double(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/*
 * [P4-code] BitLinear.forward steps 1-2 and [P4-eq] item 2, per token row t:
 *   RMSNorm:   n_k = x_k * r * g_k,  r = 1 / sqrt(mean_k(x_k^2) + rms_eps)
 *   absmax:    x_q[k] = Clip(Round(n_k * Q_b / c), -128, 127), Q_b = 127,
 *              c = max(max_k|n_k|, 1e-8)   (activation_quant clamps the max of
 *              its input, the normalized row, at 1e-8)
 *   scale:     sigma = c / Q_b   (the activation half of the dequant scale
 *              gamma * max|x| / Q_b of item 4)
 *
 * Which side of the clamp a row falls on is decided in binary32, the precision
 * of the page's code: r32 = fl(1 / fl(sqrt(fl(fl(mean x^2) + rms_eps)))) and
 * max|n| = fl(max|p| * r32), with p_k = x_k * g_k (exact in binary32: two 8-bit
 * significands).
 *
 * Rows with max|n| >= 1e-8 (every row of real activations): r > 0 is one
 * number per row, so it cancels exactly from n_k / max|n|, and the integer
 * codes are those of p_k = x_k * g_k.  127 * p_k is exact in binary64, and the
 * binary64 quotient 127 p / m (m = max|p|) can never round onto a
 * half-integer that the exact quotient is not, so rint() below returns the
 * exactly rounded code (ties to even).  sigma = m * r / 127 in binary64.
 *
 * Rows with max|n| < 1e-8 (all-zero rows, rows of tiny values, zero gains):
 * c = 1e-8 and the codes depend on r; they are formed as the page's code forms
 * x_norm * (Q_b / c), in binary32: q = rint(fl(fl(p * r32) * fl(127 / 1e-8))).
 * sigma = 1e-8 / 127.
 *
 * gain == NULL means g_k = 1; rms_eps < 0 means no RMSNorm (r = r32 = 1).
 */
void oracle_act_quant(const uint16_t *x, const uint16_t *gain, double rms_eps,
                      int64_t M, int64_t K, int8_t *xq, double *sigma)
{
    const float clampv = 1e-8f;
    int64_t t, k;
    for (t = 0; t < M; ++t) {
        const uint16_t *row = x + t * K;
        double m = 0.0, ss = 0.0;
        float r32 = 1.0f, nmax;
        for (k = 0; k < K; ++k) {
            double xv = bf16_to_double(row[k]);
            double p = gain ? xv * bf16_to_double(gain[k]) : xv;
            if (fabs(p) > m) m = fabs(p);
            ss += xv * xv;
        }
        if (rms_eps >= 0.0) {
            float ms = (float)(ss / (double)K);
            float v = ms + (float)rms_eps;
            r32 = 1.0f / sqrtf(v);
        }
        nmax = (float)m * r32;                 /* m is a binary32 value */
        if (nmax >= clampv) {
            double r = rms_eps >= 0.0 ? 1.0 / sqrt(ss / (double)K + rms_eps) : 1.0;
            for (k = 0; k < K; ++k) {
                double xv = bf16_to_double(row[k]);
                double p = gain ? xv * bf16_to_double(gain[k]) : xv;
                double v = rint(127.0 * p / m);
                if (v > 127.0) v = 127.0;
                if (v < -128.0) v = -128.0;
                xq[t * K + k] = (int8_t)v;
            }
            sigma[t] = m * r / 127.0;
        } else {
            const float sc = 127.0f / clampv;
            for (k = 0; k < K; ++k) {
                float xv = (float)bf16_to_double(row[k]);
                float p = gain ? xv * (float)bf16_to_double(gain[k]) : xv;
                float n = p * r32;
                float v = rintf(n * sc);
                if (v > 127.0f) v = 127.0f;
                if (v < -128.0f) v = -128.0f;
                xq[t * K + k] = (int8_t)v;
            }
            sigma[t] = (double)clampv / 127.0;
        }
    }
}

/* ------------------------------------------------------------------------- */
/* integer ternary contraction and dequantization                            */
/* ------------------------------------------------------------------------- */

/*
 * [P4-eq] item 3, [P3-how] item 3 and the accumulation loop of [P5-lut]:
 *   acc[t][n] = sum_k W_q[n][k] * x_q[t][k]
 * formed in int32 by adding x when the weight is +1, skipping it when 0 and
 * subtracting it when -1.  Row-major x_q [M,K], W_q [N,K], acc [M,N].
 */
void oracle_ternary_matmul(const int8_t *xq, const int8_t *wq, int64_t M, int64_t N,
                           int64_t K, int32_t *acc)
{
    int64_t t, n, k;
    for (t = 0; t < M; ++t) {
        for (n = 0; n < N; ++n) {
            int32_t a = 0;
            for (k = 0; k < K; ++k) {
                int8_t w = wq[n * K + k];
                int8_t v = xq[t * K + k];
                if (w == 1) a += v;
                else if (w == -1) a -= v;
            }
            acc[t * N + n] = a;
        }
    }
}

/* Same rule for a list of (t, n) output positions only. */
void oracle_ternary_matmul_at(const int8_t *xq, const int8_t *wq, int64_t K,
                              const int64_t *ts, const int64_t *ns, int64_t count,
                              int32_t *acc)
{
    int64_t i, k;
    for (i = 0; i < count; ++i) {
        const int8_t *xr = xq + ts[i] * K;
        const int8_t *wr = wq + ns[i] * K;
        int32_t a = 0;
        for (k = 0; k < K; ++k) {
            if (wr[k] == 1) a += xr[k];
            else if (wr[k] == -1) a -= xr[k];
        }
        acc[i] = a;
    }
}

/*
 * [P4-eq] item 4 and [P4-code] step 4: y = acc * (gamma * max|n| / Q_b), i.e.
 * y[t][n] = acc[t][n] * sigma[t] * w_scale[n], in binary64.
 */
void oracle_dequant(const int32_t *acc, const double *sigma, const double *w_scale,
                    int64_t M, int64_t N, double *y)
{
    int64_t t, n;
    for (t = 0; t < M; ++t)
        for (n = 0; n < N; ++n)
            y[t * N + n] = (double)acc[t * N + n] * sigma[t] * w_scale[n];
}

/* ------------------------------------------------------------------------- */
/* per-tensor activation quantization with Q_b = 128                         */
/* ------------------------------------------------------------------------- */

/*
 * [P5-aq] "BitNet 1-bit LLM Inference Framework", BitLinear.activation_quantize
 * (the variant of that page): one scale for the whole tensor,
 *   gamma = max_{t,k} |x|,   x_q = Round(Clip(x * Q_b / (gamma + 1e-8), -Q_b, Q_b - 1))
 * with Q_b = 2^(8-1) = 128; the clip comes before the rounding, as in the page's
 * code, so codes lie in [-128, 127]; Round is nearest, ties to even.  No
 * RMSNorm.  The page's tensors are binary32, so the quotient is formed in
 * binary32: x * 128 is exact, gamma + 1e-8 is one binary32 rounding and the
 * division one more; that rounded quotient decides the code.  The dequant
 * factor of every token is sigma = gamma / 128 (the page multiplies the
 * integer product by w_scale * gamma / 2^7).
 */
void oracle_act_quant_per_tensor(const uint16_t *x, int64_t M, int64_t K, int8_t *xq, double *sigma)
{
    int64_t i, n = M * K;
    double g = 0.0;
    float d;
    for (i = 0; i < n; ++i) {
        double a = fabs(bf16_to_double(x[i]));
        if (a > g) g = a;
    }
    d = (float)g + 1e-8f;
    for (i = 0; i < n; ++i) {
        float xs = (float)bf16_to_double(x[i]) * 128.0f;
        float t = xs / d;
        if (t < -128.0f) t = -128.0f;
        if (t > 127.0f) t = 127.0f;
        xq[i] = (int8_t)rintf(t);
    }
    for (i = 0; i < M; ++i) sigma[i] = g / 128.0;
}
