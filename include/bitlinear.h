/*
 * bitlinear.h - C ABI of the BitNet b1.58 BitLinear forward for one B300 GPU (sm_103a).
 *
 * The forward has three steps, each an entry point below:
 *   1. bitlinear_pack_weights: absmean ternarization of the latent weights and
 *      2-bit packing (done once per weight matrix);
 *   2. bitlinear_quant_act: RMSNorm + per-token absmax int8 quantization of the
 *      activations;
 *   3. bitlinear_forward: exact int32 ternary contraction of the int8 tokens with
 *      the packed weights, dequantized by gamma * max|x| / 127.
 *
 * Sources (page title, section):
 *   [P4-eq]   "BitNet b1.58 in Production: 1-Bit LLMs and Energy Benchmarks",
 *             "The Mathematical Mechanism: BitLinear vs Standard Linear", items 1-4.
 *   [P4-code] same page, "Production Multi-File Implementation", bit_linear.py
 *             (weight_quant, activation_quant, BitLinear.forward).
 *   [P5-lut]  "BitNet 1-bit LLM Inference Framework", "How the LUT Kernel Works"
 *             (2-bit code 00 = 0, 01 = +1, 10 = -1, four weights per byte;
 *             int32 accumulation, C signature (act, weight, out, M, N, K)).
 *   [P1-impl] "BitNet's 1-Bit Transformer: Architecture Breakdown", "Core
 *             Modifications", item 1 (bitlinear_forward(x, W_packed, s)).
 *
 * Conventions shared by every call:
 *   - Pointers are DEVICE pointers owned by the caller (allocated e.g. by PyTorch),
 *     16-byte aligned, row-major and densely packed.  The library allocates, frees
 *     and synchronizes nothing inside these calls; scratch memory is the caller's
 *     `workspace`, sized by the matching *_workspace_bytes function.
 *   - All work is enqueued on `stream` (a cudaStream_t passed as void*; NULL is the
 *     legacy default stream).  Results are valid once the stream has reached them.
 *   - Argument errors are reported synchronously before anything is enqueued, and
 *     then nothing is written.  A failed launch returns BITLINEAR_ERR_CUDA.  Errors
 *     found on the device (a non-finite weight, a bounded wait that ran out) are
 *     recorded in a per-device error word read by bitlinear_get_device_error.
 *   - The calling thread's current CUDA device must be an sm_103 GPU (B300), else
 *     BITLINEAR_ERR_DEVICE.  No exception crosses the ABI.
 */
#ifndef BITLINEAR_H_
#define BITLINEAR_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum bitlinear_status {
    BITLINEAR_OK = 0,
    BITLINEAR_ERR_NULL = 1,       /* a required pointer is NULL */
    BITLINEAR_ERR_SHAPE = 2,      /* a size is negative, zero where it must not be, or breaks a divisibility rule */
    BITLINEAR_ERR_ALIGN = 3,      /* a pointer is not 16-byte aligned */
    BITLINEAR_ERR_DTYPE = 4,      /* unknown out_dtype */
    BITLINEAR_ERR_DEVICE = 5,     /* current device is not sm_103, or no device */
    BITLINEAR_ERR_CUDA = 6,       /* a CUDA runtime call or launch failed */
    BITLINEAR_ERR_TIMEOUT = 7,    /* device: a bounded wait in a kernel ran out */
    BITLINEAR_ERR_WORKSPACE = 8,  /* workspace missing or smaller than required */
    BITLINEAR_ERR_NONFINITE = 9,  /* device: a latent weight was Inf or NaN */
    BITLINEAR_ERR_FLAGS = 10      /* unknown bits in a flags argument */
} bitlinear_status;

/* Output element types of bitlinear_forward. */
#define BITLINEAR_OUT_F32 0
#define BITLINEAR_OUT_BF16 1
#define BITLINEAR_OUT_BF16_ADD 2   /* y is bf16 and is updated in place: y = bf16(y + result) */

/*
 * Flag of bitlinear_quant_act and bitlinear_forward: launch the call's kernels
 * as programmatic dependents of the work already on the stream, so that they
 * start while that work finishes.  Before waiting for it, a kernel reads only
 * the packed weights and w_scale (bitlinear_forward) or nothing at all
 * (bitlinear_quant_act); so with this flag the packed weights and w_scale
 * must not be written by work still in flight on the stream.  Everything else
 * keeps plain stream order.
 */
#define BITLINEAR_FLAG_PDL 1u

/*
 * Largest token count for which bitlinear_forward, given x_q, contracts on the
 * int8 codes directly (a persistent CUDA-core kernel with int8 dot products;
 * x_ops is then not read and no workspace is needed).  It does so for M = 1
 * (every K) and M = 2 (K <= 37376), where the tokens' staged codes fit in
 * shared memory; bitlinear_forward_workspace_bytes returns 0 exactly then.
 * Otherwise, or with x_ops alone, the tensor-core kernels run on the operand
 * form.  Results are identical.
 */
#define BITLINEAR_CODES_MAX_M 2

/* Human-readable name of a status code (static string, never NULL). */
const char *bitlinear_status_string(bitlinear_status status);

/* ABI version, currently 2 (2 added the l2_prefetch arguments of bitlinear_forward
 * and bitlinear_linear_forward). */
int bitlinear_abi_version(void);

/* Number of kernels this library has enqueued in this process so far (all devices,
 * all threads; memsets not counted).  For accounting in benchmarks and tests. */
uint64_t bitlinear_kernel_launches(void);

/* ------------------------------------------------------------------------ */
/* 1. weights                                                                */
/* ------------------------------------------------------------------------ */

/* Bytes of the packed ternary matrix in the tile-major layout below: Np * Kp / 4,
 * with Np = N rounded up to a multiple of 16 and Kp = K rounded up to a multiple
 * of 512 (the padding holds zero codes); 0 for shapes bitlinear_pack_weights rejects. */
size_t bitlinear_packed_bytes(int64_t N, int64_t K);

/* Bytes of scratch that bitlinear_pack_weights needs (independent of N and K). */
size_t bitlinear_pack_workspace_bytes(int64_t N, int64_t K);

/*
 * Absmean ternarization and 2-bit packing of one latent weight matrix
 * ([P4-eq] item 1; [P4-code] weight_quant; [P5-lut] code table).
 *
 *   gamma  = (1/(N K)) sum |W|, the exact mean rounded once to binary32
 *   d      = fl32(gamma + eps)
 *   W_q    = Clip(Round(W / d), -1, 1)   (Round: nearest, ties to even)
 *
 * W        [N,K] fp32, nn.Linear layout (row n = output feature n).  Must be finite.
 * N, K     N >= 1, K >= 4, K % 4 == 0, N*K < 2^32.
 * eps      the eps of the divisor (1e-5 in BitNet b1.58); must be >= 0.
 * packed   bitlinear_packed_bytes(N,K) uint8 out.  The codes of one row form the
 *          canonical packed row: weight k in byte k/4, bits 2*(k%4)..2*(k%4)+1,
 *          code 00 = 0, 01 = +1, 10 = -1 (11 never written).  The rows are stored
 *          tile-major for the contraction kernels: rows padded to Np = N rounded
 *          up to 16 and grouped in tiles of 128 (the last tile holds the remaining
 *          Np % 128), K padded to Kp = K rounded up to 512 (segments of 128 bytes
 *          per row); within a tile of R rows each segment is one contiguous block
 *          of R x 128 bytes, and byte b of row n's canonical row sits at
 *            (n/128)*128*(Kp/512)*128 + (b/128)*R*128 + (n%128)*128
 *              + (((b%128)/16) ^ (n%8))*16 + b%16.
 *          Padding holds zero codes.  Concatenating the outputs for matrices of
 *          N_i rows gives the packing of the stacked matrix when every N_i but the
 *          last is a multiple of 128.
 * w_scale  [N] fp32 out: gamma repeated for every row (a per-row scale vector lets
 *          several matrices be stacked into one fused projection).
 * gamma_out [1] fp32 out, or NULL.
 * workspace >= bitlinear_pack_workspace_bytes(N,K) bytes of device scratch; its
 *          contents on entry do not matter (the call clears what it uses).
 * Device errors: a non-finite weight sets BITLINEAR_ERR_NONFINITE in the device
 *          error word; the outputs are then unspecified.
 */
bitlinear_status bitlinear_pack_weights(const float *W, int64_t N, int64_t K, float eps,
                                        uint8_t *packed, float *w_scale, float *gamma_out,
                                        void *workspace, size_t workspace_bytes, void *stream);

/*
 * bitlinear_pack_weights without a workspace argument: the same kernels and the
 * same results, with the ~2 KB of scratch taken from a fixed array that the
 * library keeps in each GPU's memory.  The pages have no counterpart to this
 * call; it is here for callers that cannot allocate device memory, such as a
 * plugin that is only handed buffers its host framework sized in advance, or
 * code on a latency-critical path where cudaMalloc/cudaFree may synchronize the
 * device or fail under memory pressure.  The call itself allocates nothing.
 *
 * Arguments, layouts and device errors: as bitlinear_pack_weights.
 * Limit: N*K < 2^32 (else BITLINEAR_ERR_SHAPE); the fixed scratch holds
 *   bitlinear_pack_workspace_bytes() bytes, which covers every size within it.
 * The first call on each device looks up the array's device address with that
 *   device current, so make it before any stream capture.
 * Every GPU that loads the library holds the array until the process exits.
 * All calls on a device share the one array and leave their contents in it;
 *   each call clears what it accumulates into, but calls whose work overlaps on
 *   the GPU (unordered streams) race on it: order them.
 */
bitlinear_status bitlinear_pack_weights_static(const float *W, int64_t N, int64_t K, float eps,
                                               uint8_t *packed, float *w_scale, float *gamma_out,
                                               void *stream);

/*
 * Ternarization with a scale per output channel ([P2-wr] "BitNet-2B-4T:
 * Inside the 2B-Parameter, 4T-Token 1-Bit LLM", section "Weight
 * Representation: Ternary + Scale, Not Pure Binary": W_bit x s, s in R^d):
 * the absmean of [P4-eq] item 1 taken over each row,
 *
 *   gamma_n  = (1/K) sum_k |W[n][k]|, the exact row mean rounded once to binary32
 *   W_q[n]   = Clip(Round(W[n] / fl32(gamma_n + eps)), -1, 1)
 *
 * and w_scale[n] = gamma_n, which bitlinear_forward applies per output row.
 * (The page stores s in FP16; w_scale stays binary32 here.)
 * W, N, K, eps, packed, device errors: as bitlinear_pack_weights.
 * w_scale  [N] fp32 out: gamma_n.
 * Needs no scratch.
 */
bitlinear_status bitlinear_pack_weights_per_channel(const float *W, int64_t N, int64_t K, float eps,
                                                    uint8_t *packed, float *w_scale, void *stream);

/* ------------------------------------------------------------------------ */
/* 2. activations                                                            */
/* ------------------------------------------------------------------------ */

/*
 * Bytes of the tensor-core operand form of M tokens of K int8 codes ("x_ops"):
 * 2 * Mt * Kp with Kp = K rounded up to a multiple of 512 and Mt = M rounded up
 * to a multiple of 8 for M <= 32 (decode), to a multiple of 256 above (prefill).
 * Each code x is kept as two e4m3 planes, 16*floor((x+8)/16) and the remainder
 * in [-8, 7], in the swizzled shared-memory layout the tensor cores read; it is
 * an internal format that only bitlinear_forward reads, and it depends on M, so
 * x_ops written for M tokens is only valid for a forward with the same M.
 */
size_t bitlinear_act_ops_bytes(int64_t M, int64_t K);

/*
 * RMSNorm + per-token absmax int8 quantization ([P4-code] BitLinear.forward
 * steps 1-2 and activation_quant; [P4-eq] item 2, Q_b = 127), one token per row:
 *
 *   n_k    = x_k * r * g_k,  r = 1/sqrt(mean_k x_k^2 + rms_eps)      (RMSNorm)
 *   x_q[k] = Clip(Round(127 * n_k / max_k|n_k|), -128, 127)          (Round: ties to even)
 *   act_scale = max_k|n_k| / 127                                      (sigma, the per-token dequant factor)
 *
 * Because r > 0 is one number per row, x_q equals the codes of x*g computed
 * exactly: the kernel decides every code from exact binary32 products, so x_q is
 * bit-exact whatever the summation order of mean(x^2).  As activation_quant
 * clamps its scale, a row whose max|n_k| (formed as fl32(max|x*g| * r), r =
 * fl32(1 / fl32(sqrt(fl32(fl32(mean x^2) + rms_eps))))) is below 1e-8 uses 1e-8 as
 * its max: its codes are rint(fl32(fl32(x g r) * fl32(127 / 1e-8))) and act_scale
 * = 1e-8 / 127 (all-zero rows give zero codes).
 *
 * x_bf16   [M,K] bf16 tokens.  Must be finite, with |x| <= 2^60 and |x*g| <= 2^100
 *          (beyond that the fp32 squares or products may overflow).
 * gain_bf16 [K] bf16 RMSNorm weight g, or NULL for g = 1.
 * rms_eps  eps of RMSNorm (>= 0); a negative value disables RMSNorm (r = 1).
 * M, K     M >= 0 (M == 0 enqueues nothing and accepts NULL buffers), 8 <= K <= 65536,
 *          K % 8 == 0.
 * x_q      [M,K] int8 out.  act_scale [M] fp32 out.
 * x_ops    bitlinear_act_ops_bytes(M,K) bytes out (the same codes in the operand
 *          form that bitlinear_forward consumes), or NULL.  Passing it lets
 *          several forwards share one conversion.
 * flags    0 or BITLINEAR_FLAG_PDL.
 */
bitlinear_status bitlinear_quant_act(const void *x_bf16, const void *gain_bf16, float rms_eps,
                                     int64_t M, int64_t K, int8_t *x_q, float *act_scale,
                                     void *x_ops, unsigned flags, void *stream);

/* Bytes of scratch that bitlinear_quant_act_per_tensor needs (4 M, rounded up). */
size_t bitlinear_quant_act_per_tensor_workspace_bytes(int64_t M);

/*
 * Per-tensor absmax quantization with Q_b = 128 ([P5-aq] "BitNet 1-bit LLM
 * Inference Framework", BitLinear.activation_quantize), the scale-granularity
 * variant of bitlinear_quant_act: one scale for all M x K values and no RMSNorm,
 *
 *   gamma    = max_{t,k} |x[t][k]|
 *   x_q[t,k] = Round(Clip(fl32(fl32(x * 128) / fl32(gamma + 1e-8)), -128, 127))
 *   act_scale[t] = gamma / 128                     (the same for every token)
 *
 * The clip comes before the rounding, as in the page's code, so codes span
 * [-128, 127]; the quotient is rounded once to binary32 before Round (ties to
 * even), so the codes are exact given that quotient.  bitlinear_forward accepts
 * these codes and scales unchanged (y = acc * gamma / 128 * w_scale).
 *
 * x_bf16, M, K, x_q, act_scale, x_ops, flags: as bitlinear_quant_act.
 * workspace >= bitlinear_quant_act_per_tensor_workspace_bytes(M) bytes of device
 *           scratch (the row maxima); contents on entry do not matter.
 */
bitlinear_status bitlinear_quant_act_per_tensor(const void *x_bf16, int64_t M, int64_t K, int8_t *x_q,
                                                float *act_scale, void *x_ops, void *workspace,
                                                size_t workspace_bytes, unsigned flags, void *stream);

/* ------------------------------------------------------------------------ */
/* 3. ternary contraction + dequantization                                   */
/* ------------------------------------------------------------------------ */

/* Bytes of scratch that bitlinear_forward needs for this shape when it is called
 * with x_ops == NULL (it then converts x_q into the workspace first); 0 when the
 * int8-code kernel takes x_q (see BITLINEAR_CODES_MAX_M).  Called with x_ops, it
 * needs none. */
size_t bitlinear_forward_workspace_bytes(int64_t M, int64_t N, int64_t K);

/*
 * y = dequant(x_q . W_q^T) ([P4-eq] items 3-4; [P5-lut] accumulation loop;
 * [P1-impl] bitlinear_forward(x, W_packed, s)):
 *
 *   acc[t][n] = sum_k W_q[n][k] * x_q[t][k]                 exact, int32
 *   y[t][n]   = fl32(fl32(acc * act_scale[t]) * w_scale[n]) then, for bf16
 *               output, rounded to nearest even bf16.
 *
 * x_q       [M,K] int8 (from bitlinear_quant_act or bitlinear_quant_act_per_tensor).
 *           Codes may be any int8 in [-128, 127].
 *           May be NULL when x_ops is given.
 * act_scale [M] fp32.
 * x_ops     the same codes in operand form (bitlinear_quant_act's x_ops), or NULL.
 *           With x_q given and M <= BITLINEAR_CODES_MAX_M it is not read.
 * packed    [N,K/4] uint8 (from bitlinear_pack_weights).
 * w_scale   [N] fp32.
 * M, N, K   0 <= M <= 2^24 (M == 0 enqueues nothing and accepts NULL buffers),
 *           16 <= N <= 2^24, N % 16 == 0, 128 <= K <= 65536, K % 128 == 0.
 * out_dtype BITLINEAR_OUT_F32, BITLINEAR_OUT_BF16, or BITLINEAR_OUT_BF16_ADD (residual
 *           connection: y holds bf16 values on entry and receives bf16(fl32(y) + result)).
 * y         [M,N] out, fp32 or bf16.
 * acc_debug [M,N] int32 out with the raw accumulators, or NULL (for parity checks).
 * workspace >= bitlinear_forward_workspace_bytes(M,N,K) bytes of device scratch
 *           when x_ops is NULL (may be NULL when that is 0, or with x_ops).
 *           Contents on entry do not matter.
 * l2_prefetch, l2_prefetch_bytes  a range of device memory of the current
 *           device (16-byte aligned; the size is rounded down to 16 bytes), or
 *           NULL / 0: typically the packed weights of the call that follows on
 *           the stream.  The decode kernels (M <= 32) ask the copy engine to
 *           pull it into L2 while they run, so that a chain of decode calls
 *           keeps HBM streaming weights across its launches; the prefill
 *           contraction ignores it.  It is a cache hint only: the range is not
 *           read otherwise, results do not depend on it, and it may be written
 *           by other work at any time.
 * flags     0 or BITLINEAR_FLAG_PDL.
 *
 * Exactness: every route forms acc as the exact integer sum.  With x_q given and
 * M <= BITLINEAR_CODES_MAX_M (see there for the exact shape rule) a CUDA-core
 * kernel contracts the int8 codes with int32 dot products (|acc| <= 128 K < 2^31).
 * Otherwise the tensor cores contract e4m3 operands: each code enters as two
 * exact e4m3 values (see bitlinear_act_ops_bytes) and every fp32 accumulator
 * stays an integer below 2^24 in magnitude (at most 128 K <= 2^23).  Both give
 * the same acc and y bit for bit.
 */
bitlinear_status bitlinear_forward(const int8_t *x_q, const float *act_scale, const void *x_ops,
                                   const uint8_t *packed, const float *w_scale,
                                   int64_t M, int64_t N, int64_t K, int out_dtype, void *y,
                                   int32_t *acc_debug, void *workspace, size_t workspace_bytes,
                                   const void *l2_prefetch, size_t l2_prefetch_bytes,
                                   unsigned flags, void *stream);

/* Bytes of scratch that bitlinear_linear_forward needs: the operand form of the
 * codes and the per-token scales. */
size_t bitlinear_linear_workspace_bytes(int64_t M, int64_t N, int64_t K);

/* Which kernels bitlinear_linear_forward launches for this shape (the results do
 * not depend on it):
 *   BITLINEAR_ROUTE_FUSED    one kernel: RMSNorm, quantization and the int8-code
 *                            contraction together (one token, K <= 8192, or
 *                            K <= 16384 for at least 12 MiB of packed weights);
 *   BITLINEAR_ROUTE_CODES    quantization to int8 codes, then the CUDA-core
 *                            contraction on them (one token with longer K, or
 *                            two tokens);
 *   BITLINEAR_ROUTE_DECODE   quantization to the operand form, then the tcgen05
 *                            decode contraction (3 to 32 tokens, or two where
 *                            their codes do not fit the CUDA-core kernel);
 *   BITLINEAR_ROUTE_PREFILL  quantization to the operand form, then the tcgen05
 *                            prefill contraction (more tokens).
 * -1 for shapes the call rejects. */
#define BITLINEAR_ROUTE_FUSED 0
#define BITLINEAR_ROUTE_CODES 1
#define BITLINEAR_ROUTE_DECODE 2
#define BITLINEAR_ROUTE_PREFILL 3
int bitlinear_linear_route(int64_t M, int64_t N, int64_t K);

/*
 * CTAs per thread-block cluster that the prefill contraction (the
 * BITLINEAR_ROUTE_PREFILL kernel of bitlinear_forward and
 * bitlinear_linear_forward) uses for operands at x_ops: 2 when x_ops is device
 * memory of the calling thread's current device and N spans at least two
 * 128-row weight blocks, 1 otherwise.  With 2, one copy of each activation block
 * from x_ops is multicast to both CTAs of the cluster; the check keeps such
 * copies to this GPU's own memory (host, managed or peer memory is never their
 * source).  -1 when the shape does not take the prefill route or x_ops is NULL.
 * The result depends only on the arguments and the current device; nothing is
 * enqueued.
 */
int bitlinear_prefill_cluster_size(const void *x_ops, int64_t M, int64_t N, int64_t K);

/*
 * The whole BitLinear layer in one call ([P4-code] BitLinear.forward: RMSNorm,
 * activation_quant, the ternary product and the rescale; [P1-impl]
 * bitlinear_forward(x, W_packed, s)).  For one token with K <= 8192 (K <= 16384
 * for at least 12 MiB of packed weights) a single kernel does all of it
 * (BITLINEAR_ROUTE_FUSED); otherwise the call enqueues
 * bitlinear_quant_act into the workspace (int8 codes or the operand form), then
 * bitlinear_forward on it, the second launch overlapping the first (programmatic
 * dependent launch).  bitlinear_linear_route tells which.  Results equal those of
 * the two calls bit for bit.
 *
 * x_bf16, gain_bf16, rms_eps  as bitlinear_quant_act (K % 128 == 0 here).
 * packed, w_scale, M, N, K, out_dtype, y, acc_debug  as bitlinear_forward.
 * x_q       [M,K] int8 out, or NULL.  act_scale [M] fp32 out, or NULL (then kept
 *           in the workspace).
 * workspace >= bitlinear_linear_workspace_bytes(M,N,K) bytes of device scratch
 *           (required on every route; the one-kernel route leaves it untouched).
 *           Contents on entry do not matter.
 * l2_prefetch, l2_prefetch_bytes  as bitlinear_forward (the next call's weights,
 *           or NULL / 0); the contraction kernel issues it.
 * flags     0 or BITLINEAR_FLAG_PDL (the first launch may overlap the work
 *           already on the stream).
 */
bitlinear_status bitlinear_linear_forward(const void *x_bf16, const void *gain_bf16, float rms_eps,
                                          const uint8_t *packed, const float *w_scale, int64_t M,
                                          int64_t N, int64_t K, int out_dtype, void *y, int8_t *x_q,
                                          float *act_scale, int32_t *acc_debug, void *workspace,
                                          size_t workspace_bytes, const void *l2_prefetch,
                                          size_t l2_prefetch_bytes, unsigned flags, void *stream);

/* ------------------------------------------------------------------------ */
/* 4. the linear stack of a BitNet b1.58 transformer                         */
/* ------------------------------------------------------------------------ */

/*
 * One layer's BitLinear weights (device pointers, packed by
 * bitlinear_pack_weights) and RMSNorm gains (bf16, device).  Every BitLinear
 * has its own RMSNorm before its activation quantization ([P4-code]
 * BitLinear.forward).  gate_up stacks the gate rows (0..F-1) above the up rows
 * (F..2F-1), each matrix with its own gamma in gate_up_scale.
 */
typedef struct bitlinear_layer {
    const uint8_t *qkv;     const float *qkv_scale;      /* NQKV x H  */
    const uint8_t *o;       const float *o_scale;        /* H x H     */
    const uint8_t *gate_up; const float *gate_up_scale;  /* 2F x H    */
    const uint8_t *down;    const float *down_scale;     /* H x F     */
    const void *gain_qkv;   /* bf16 [H] */
    const void *gain_o;     /* bf16 [H] */
    const void *gain_gate_up; /* bf16 [H] */
    const void *gain_down;  /* bf16 [F] */
} bitlinear_layer;

/* Bytes of scratch that bitlinear_block_forward needs. */
size_t bitlinear_block_workspace_bytes(int64_t M, int64_t H, int64_t NQKV, int64_t F);

/*
 * Bytes of one layer's trace of bitlinear_block_forward (see its `trace`
 * argument).  The layer's trace holds, each part starting 256-byte aligned, in
 * this order: the int8 codes of the inputs of its four BitLinears (qkv, o,
 * gate_up: [M, H]; down: [M, F]), their token scales ([4][M] fp32), qkv
 * ([M, NQKV] bf16), x after the O residual ([M, H] bf16), gate|up ([M, 2F]
 * fp32) and x after the down residual ([M, H] bf16).
 */
size_t bitlinear_block_trace_bytes(int64_t M, int64_t H, int64_t NQKV, int64_t F);

/*
 * The BitLinear projections of n_layers transformer layers on M tokens, with
 * x [M, H] bf16 (device) as the residual stream, updated in place.  Per layer
 * (every "BitLinear" = RMSNorm + int8 quantization + ternary contraction +
 * dequantization, as bitlinear_quant_act + bitlinear_forward):
 *
 *   qkv = BitLinear_qkv(x)                  fp32 [M, NQKV], kept as bf16
 *   q   = qkv[:, 0:H]                       attention is not part of this
 *                                           library: the query slice stands in
 *                                           for the attention output
 *   x   = bf16(x + BitLinear_o(q))
 *   g|u = BitLinear_gate_up(x)              fp32 [M, 2F]
 *   h   = bf16(fl(fl(max(g, 0)^2) * u))     ReLU^2 gating
 *   x   = bf16(x + BitLinear_down(h))
 *
 * Sources: [P4-code] BitLinear.forward (RMSNorm inside every BitLinear);
 * [P5-block] "BitNet 1-bit LLM Inference Framework", section "A Full BitNet
 * Transformer Block" (q/k/v/o and gate/up/down BitLinear projections, residual
 * adds around attention and FFN).  The FFN gate here is squared ReLU, the
 * activation of the 2B-parameter BitNet b1.58 models, in place of that block's
 * SiLU; the block's LayerNorms are the RMSNorms of the BitLinears.
 *
 * layers    HOST array of n_layers structs holding device pointers.
 * H, NQKV, F  hidden size, QKV width (>= H), FFN width; H and F multiples of 128,
 *           NQKV a multiple of 16.
 * rms_eps   eps of every RMSNorm (>= 0).
 * M         tokens, 1 <= M <= 2^20.
 * workspace >= bitlinear_block_workspace_bytes(M, H, NQKV, F) bytes of device
 *           scratch, 256-byte aligned; contents on entry do not matter.
 * trace     NULL, or n_layers * bitlinear_block_trace_bytes(M, H, NQKV, F) bytes
 *           (trace_bytes) of device memory, 256-byte aligned, that receives
 *           every layer's intermediates (layout at bitlinear_block_trace_bytes)
 *           for checking each BitLinear on its exact input.  Tracing adds four
 *           small copy kernels per layer; the results are the same.
 * flags     0 or BITLINEAR_FLAG_PDL (applies to the first kernel; the
 *           following ones always overlap with their predecessor).
 * Every contraction pulls the packed weights of the projection after it into L2
 * (see the l2_prefetch argument of bitlinear_forward).
 */
bitlinear_status bitlinear_block_forward(const bitlinear_layer *layers, int n_layers, int64_t H,
                                         int64_t NQKV, int64_t F, float rms_eps, void *x_bf16,
                                         int64_t M, void *workspace, size_t workspace_bytes,
                                         void *trace, size_t trace_bytes, unsigned flags, void *stream);

/* ------------------------------------------------------------------------ */
/* device error word                                                         */
/* ------------------------------------------------------------------------ */

/*
 * Waits for `stream`, then returns and clears the current device's error word:
 * BITLINEAR_OK if no kernel of this library recorded an error since the last
 * call, else the first recorded device status (BITLINEAR_ERR_TIMEOUT,
 * BITLINEAR_ERR_NONFINITE).  Returns BITLINEAR_ERR_CUDA if the wait or the read
 * fails.  This is the only call that synchronizes.
 */
bitlinear_status bitlinear_get_device_error(void *stream);

#ifdef __cplusplus
}
#endif

#endif /* BITLINEAR_H_ */
