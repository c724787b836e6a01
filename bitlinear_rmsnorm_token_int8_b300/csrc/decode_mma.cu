// Decode contraction (few tokens): y = dequant(x_q . W_q^T), streaming the
// 2-bit packed weights from HBM through shared memory and contracting them on
// the tensor cores with mma.sync m16n8k32 e4m3, exact in fp32 (act_ops.cuh
// explains the two-plane split of the int8 codes).
//
// Page "BitNet b1.58 in Production: 1-Bit LLMs and Energy Benchmarks", section
// "The Mathematical Mechanism", items 3-4 (integer accumulation of the ternary
// products, dequantization by gamma * max|x| / Q_b); page "BitNet 1-bit LLM
// Inference Framework", section "How the LUT Kernel Works" (2-bit code
// 00 = 0, 01 = +1, 10 = -1, four weights per byte, int32 accumulation).
//
// Structure: a persistent grid, one CTA per SM.  Work items are
// (token tile of <= 16, group of T row tiles of 16 rows = R rows, all of K);
// CTA c takes items c, c + gridDim.x, ...  Warp 0 is the producer.  A stage is
// SBK segments of 512 k: per row tile one bulk copy of the tile's SBK
// contiguous 2 KB blocks of the tile-major packed layout, plus one bulk copy
// of the activation operands of those segments; stages go through a ring of
// NS slots signalled by mbarriers.  (Few, large requests matter: the copy
// engine's rate is bounded per request, ~1 TB/s for 256-byte copies against
// ~6 TB/s for 16 KB ones on this GPU, and a tensor-map box of R rows x 128
// bytes costs about as much as R small requests.)  Warps 1..C are consumers
// (C = 2 SBK, SBK a divisor of the segment count, at most 14 or 8 with two
// token tiles; a stage holds one unit per consumer): a segment is split in two units of 256 k, consumer w takes units
// w, w + C, ... of a stage, keeps a unit's activation fragments in registers
// and runs them against all T row tiles, so the T tiles share one operand
// load.  At the end of an item the consumers add their partial sums into
// shared memory as int32 (exact), then write the dequantized outputs.
//
// Weight decode.  Within a segment thread t of a quad owns k in
// [128 t, 128 t + 128), read as two 16-byte chunks (2t and 2t+1 of the row's
// 128 bytes; the packed layout stores chunk c of row r at c ^ (r % 8), so the
// two rows g, g+1 that share a shared-memory phase hit chunks of opposite
// parity: no bank conflicts).  A chunk is four 32-bit words of 16 codes, LSB first.  w & 0x33333333 leaves
// the codes of the even k in the low two bits of each nibble and
// (w >> 2) & 0x33333333 those of the odd k; each nibble then selects a byte of
// {0x00, 0x38, 0xB8} = e4m3 {0, +1, -1} through a byte permute, so four
// weights cost one PRMT.  The k order this gives inside a register
// (0,2,4,6 | 8..14 | 1,3,5,7 | 9..15) is the order of the operand layout.
//
// Exactness of the fp32 accumulation: one unit adds at most 127 * 256 in
// magnitude to an accumulator; every 16 units a warp moves its accumulators to
// int32, so an fp32 partial sum never exceeds 127 * 4096 < 2^19.
//
// Overlap (BITLINEAR_FLAG_PDL): the producer issues the weight copies of the
// first NS stages before it waits for the previous kernel; only the operand
// copies and the output stores wait for it.
//
// Bounded waits: every mbarrier wait gives up after kSpinLimit polls, records
// BITLINEAR_ERR_TIMEOUT in the device error word and makes the CTA stop work;
// before it exits, the producer waits (bounded again) for the copies it issued.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "act_ops.cuh"
#include "device_util.cuh"
#include "internal.h"

namespace bitlinear {
namespace {

constexpr uint32_t kCodeToE4M3 = 0x00B83800u;  // bytes 0x00 (code 0), 0x38 (+1), 0xB8 (-1), 0x00
constexpr int kDrainUnits = 16;
constexpr uint32_t kSpinLimit = 1u << 24;
constexpr int kMaxStages = 16;

struct DecodeParams {
  const uint8_t* packed;
  const uint8_t* x_ops;
  const float* act_scale;
  const float* w_scale;
  void* y;
  int32_t* acc_debug;
  int* dev_err;
  int M, N, K, out_dtype;
  int groups, ztiles, items;
  int nseg;                       // 512-wide k segments (K rounded up)
  int SBK, NS, stage_w_bytes, stage_bytes;
  int bres_bytes;                 // > 0: all operands resident in shared memory (one copy)
};

__device__ __forceinline__ void mma_e4m3(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t word(const uint4& v, int j) {
  return j == 0 ? v.x : j == 1 ? v.y : j == 2 ? v.z : v.w;
}

struct ItemInfo {
  int z, Mz, r0, ntiles;
};

template <int T>
__device__ __forceinline__ ItemInfo item_info(const DecodeParams& p, int item) {
  ItemInfo f;
  f.z = item / p.groups;
  const int gi = item - f.z * p.groups;
  f.Mz = min(16, p.M - 16 * f.z);
  f.r0 = gi * T * 16;
  f.ntiles = min(T, (p.N >> 4) - gi * T);
  return f;
}

// Consumer warps: blockDim.x / 32 - 1, at most CMAX.  mma.sync needs many
// warps in flight per SM (its issue cost is ~22 cycles per m16n8k32 e4m3 per
// sub-partition on this GPU).
template <int T, int MT, int CMAX>
__global__ void __launch_bounds__(32 * (1 + CMAX), 1) decode_mma_kernel(const DecodeParams p) {
  const int kConsumers = (int)(blockDim.x >> 5) - 1;
  extern __shared__ uint8_t smem_raw[];
  constexpr int R = T * 16;
  uint8_t* smem = smem_raw + ((128 - (smem_u32(smem_raw) & 127)) & 127);
  const uint32_t bres = smem_u32(smem) + p.NS * p.stage_bytes;                   // resident operands
  int* s_acc = reinterpret_cast<int*>(smem + p.NS * p.stage_bytes + p.bres_bytes);  // [16][R]
  uint64_t* bars = reinterpret_cast<uint64_t*>(s_acc + 16 * R);           // full[16], empty[16], bfull
  volatile int* s_abort = reinterpret_cast<volatile int*>(bars + 2 * kMaxStages + 1);
  const uint32_t bfull = smem_u32(bars + 2 * kMaxStages);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t ring = smem_u32(smem);
  const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + kMaxStages);
  const int nst = (p.nseg + p.SBK - 1) / p.SBK;             // stages per item

  if (threadIdx.x == 0) {
    for (int s = 0; s < p.NS; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, kConsumers);
    }
    mbar_init(bfull, 1);
    *s_abort = 0;
    fence_mbar_init();
  }
  for (int e = threadIdx.x; e < 16 * R; e += blockDim.x) s_acc[e] = 0;
  __syncthreads();
  pdl_launch_dependents();

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane != 0) return;          // one thread issues everything (few, large requests)
    const uint64_t pol = policy_evict_first();
    const int64_t Kp = (int64_t)p.nseg * 512;
    int q = 0;                      // global stage counter
    bool waited = false;
    int deferred = 0;               // stages whose operand copy waits for the previous kernel
    auto issue_ops = [&](int qq) {
      if (p.bres_bytes) return;                     // operands are staged once, resident
      const int item = blockIdx.x + (qq / nst) * gridDim.x, st = qq % nst;
      const ItemInfo f = item_info<T>(p, item);
      const int seg0 = st * p.SBK, nsg = min(p.SBK, p.nseg - seg0);
      const int slot = qq % p.NS;
      const uint8_t* src = p.x_ops + 32 * Kp * f.z + (int64_t)seg0 * 1024 * f.Mz;
      bulk_g2s(ring + slot * p.stage_bytes + p.stage_w_bytes, src, (uint32_t)(nsg * 1024 * f.Mz),
               full0 + 8 * slot);
    };
    for (int item = blockIdx.x; item < p.items && !*s_abort; item += gridDim.x) {
      const ItemInfo f = item_info<T>(p, item);
      for (int st = 0; st < nst; ++st, ++q) {
        const int slot = q % p.NS, round = q / p.NS;
        if (round >= 1) {
          if (!waited) {            // ring full: from here on the operands are needed
            pdl_wait();
            waited = true;
            if (p.bres_bytes) {
              mbar_arrive_expect_tx(bfull, (uint32_t)p.bres_bytes);
              bulk_g2s(bres, p.x_ops, (uint32_t)p.bres_bytes, bfull);
            }
            for (int d = 0; d < deferred; ++d) issue_ops(q - deferred + d);
            deferred = 0;
          }
          if (!mbar_wait_bounded(empty0 + 8 * slot, (round - 1) & 1, kSpinLimit)) {
            atomicCAS(p.dev_err, 0, kDevErrTimeout);
            *s_abort = 1;
            break;
          }
        }
        const int seg0 = st * p.SBK, nsg = min(p.SBK, p.nseg - seg0);
        const uint32_t tx = (uint32_t)(f.ntiles * nsg * 2048 + (p.bres_bytes ? 0 : nsg * 1024 * f.Mz));
        mbar_arrive_expect_tx(full0 + 8 * slot, tx);
        const uint32_t dst = ring + slot * p.stage_bytes;
        const int tile0 = f.r0 >> 4;
        for (int i = 0; i < f.ntiles; ++i)
          bulk_g2s_hint(dst + i * p.SBK * 2048, p.packed + ((int64_t)(tile0 + i) * p.nseg + seg0) * 2048,
                        (uint32_t)(nsg * 2048), full0 + 8 * slot, pol);
        if (waited) issue_ops(q);
        else ++deferred;
      }
    }
    if (!waited) {
      pdl_wait();
      if (p.bres_bytes) {
        mbar_arrive_expect_tx(bfull, (uint32_t)p.bres_bytes);
        bulk_g2s(bres, p.x_ops, (uint32_t)p.bres_bytes, bfull);
      }
      for (int d = 0; d < deferred; ++d) issue_ops(q - deferred + d);
    }
    if (p.bres_bytes && !mbar_wait_bounded(bfull, 0, kSpinLimit)) atomicCAS(p.dev_err, 0, kDevErrTimeout);
    // No copy may still be landing in shared memory when the CTA exits: wait
    // (bounded) for the last phase of every slot that was used.
    const int used = q < p.NS ? q : p.NS;
    for (int s = 0; s < used; ++s) {
      const int last = q - 1 - ((q - 1 - s) % p.NS);           // last stage issued into slot s
      if (!mbar_wait_bounded(full0 + 8 * s, (last / p.NS) & 1, kSpinLimit))
        atomicCAS(p.dev_err, 0, kDevErrTimeout);
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  // NA independent accumulators per (tile, token tile): the MMAs of one unit
  // are spread over NA * T chains so that they issue back to back instead of
  // waiting on each other's results.  (plane, parity) -> chain: NA = 4 keeps
  // all four apart, NA = 2 separates the planes.
  constexpr int NA = (T >= 4 || MT == 2) ? 2 : 4;
  pdl_wait();                        // act_scale and y follow the stream order
  if (p.bres_bytes && !mbar_wait_bounded(bfull, 0, kSpinLimit)) {
    if (lane == 0) {
      atomicCAS(p.dev_err, 0, kDevErrTimeout);
      *s_abort = 1;
    }
  }
  const int cw = warp - 1;
  const int g = lane >> 2, t = lane & 3;
  int q = 0;
  for (int item = blockIdx.x; item < p.items; item += gridDim.x) {
    const ItemInfo f = item_info<T>(p, item);
    float acc[T][MT][NA][4];
#pragma unroll
    for (int i = 0; i < T; ++i)
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int a = 0; a < NA; ++a)
#pragma unroll
          for (int c = 0; c < 4; ++c) acc[i][mt][a][c] = 0.0f;
    auto drain = [&]() {
#pragma unroll
      for (int i = 0; i < T; ++i)
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            int v = 0;
#pragma unroll
            for (int a = 0; a < NA; ++a) {
              v += __float2int_rn(acc[i][mt][a][c]);
              acc[i][mt][a][c] = 0.0f;
            }
            if (v != 0) atomicAdd(&s_acc[(mt * 8 + 2 * t + (c & 1)) * R + i * 16 + g + (c >> 1) * 8], v);
          }
    };
    // Prefetch the scales of this thread's first outputs of the item: the loads
    // complete during the contraction instead of stalling the epilogue.
    constexpr int NPF = 4;
    const int nout = f.Mz * R;
    float pf_ws[NPF], pf_as[NPF];
#pragma unroll
    for (int j = 0; j < NPF; ++j) {
      const int e = (int)threadIdx.x - 32 + j * 32 * kConsumers;
      pf_ws[j] = 0.0f;
      pf_as[j] = 0.0f;
      if (e < nout) {
        const int mm = e / R, rr = e - mm * R;
        if (rr < f.ntiles * 16) {
          pf_ws[j] = __ldg(p.w_scale + f.r0 + rr);
          pf_as[j] = __ldg(p.act_scale + 16 * f.z + mm);
        }
      }
    }
    int since_drain = 0;
    bool aborted = false;
    for (int st = 0; st < nst; ++st, ++q) {
      const int slot = q % p.NS, round = q / p.NS;
      if (!mbar_wait_bounded(full0 + 8 * slot, round & 1, kSpinLimit)) {
        if (lane == 0) {
          atomicCAS(p.dev_err, 0, kDevErrTimeout);
          *s_abort = 1;
        }
        aborted = true;
        break;
      }
      const int seg0 = st * p.SBK, nsg = min(p.SBK, p.nseg - seg0);
      const uint32_t wbase = ring + slot * p.stage_bytes;
      // operands of unit u of the item: resident block, or this stage's copy
      const uint32_t bbase = p.bres_bytes ? bres + (uint32_t)(2 * seg0) * 512 * f.Mz : wbase + p.stage_w_bytes;
      for (int cu = cw; cu < 2 * nsg; cu += kConsumers) {
        const int sg = cu >> 1, h = cu & 1;
        uint4 xb[8][MT];
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
          for (int mt = 0; mt < MT; ++mt) {
            const int m = mt * 8 + g;
            xb[i][mt] = m < f.Mz ? lds128(bbase + (uint32_t)(((cu * 8 + i) * f.Mz + m) * 4 + t) * 16)
                                 : make_uint4(0u, 0u, 0u, 0u);
          }
        // row g of a 2 KB block: 128-byte line, chunk (2t+h) stored at (2t+h) ^ g
        const uint32_t wrow = wbase + (uint32_t)(sg * 2048 + g * 128 + ((((2 * t + h) ^ g)) << 4));
        uint4 wv[T][2];
#pragma unroll
        for (int i = 0; i < T; ++i) {
          if (i < f.ntiles) {
            wv[i][0] = lds128(wrow + i * p.SBK * 2048);
            wv[i][1] = lds128(wrow + i * p.SBK * 2048 + 8 * 128);
          } else {
            wv[i][0] = make_uint4(0u, 0u, 0u, 0u);
            wv[i][1] = make_uint4(0u, 0u, 0u, 0u);
          }
        }
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
#pragma unroll
          for (int i = 0; i < T; ++i) {
            if (i < f.ntiles) {
              const uint32_t w0 = word(wv[i][0], jj), w1 = word(wv[i][1], jj);
              const uint32_t lo0 = w0 & 0x33333333u, hi0 = (w0 >> 2) & 0x33333333u;
              const uint32_t lo1 = w1 & 0x33333333u, hi1 = (w1 >> 2) & 0x33333333u;
              const uint32_t e00 = __byte_perm(kCodeToE4M3, 0u, lo0);        // row g:   k 0,2,4,6
              const uint32_t e01 = __byte_perm(kCodeToE4M3, 0u, lo0 >> 16);  //          k 8..14 even
              const uint32_t e02 = __byte_perm(kCodeToE4M3, 0u, hi0);        //          k 1,3,5,7
              const uint32_t e03 = __byte_perm(kCodeToE4M3, 0u, hi0 >> 16);  //          k 9..15 odd
              const uint32_t e10 = __byte_perm(kCodeToE4M3, 0u, lo1);        // row g+8
              const uint32_t e11 = __byte_perm(kCodeToE4M3, 0u, lo1 >> 16);
              const uint32_t e12 = __byte_perm(kCodeToE4M3, 0u, hi1);
              const uint32_t e13 = __byte_perm(kCodeToE4M3, 0u, hi1 >> 16);
#pragma unroll
              for (int mt = 0; mt < MT; ++mt) {
                const uint4 ev = xb[2 * jj][mt], od = xb[2 * jj + 1][mt];
                mma_e4m3(acc[i][mt][0], e00, e10, e01, e11, ev.x, ev.y);           // 16 h, even k
                mma_e4m3(acc[i][mt][1], e00, e10, e01, e11, ev.z, ev.w);           // l, even k
                mma_e4m3(acc[i][mt][NA == 4 ? 2 : 0], e02, e12, e03, e13, od.x, od.y);  // 16 h, odd k
                mma_e4m3(acc[i][mt][NA == 4 ? 3 : 1], e02, e12, e03, e13, od.z, od.w);  // l, odd k
              }
            }
          }
        }
        if (++since_drain == kDrainUnits) {
          drain();
          since_drain = 0;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty0 + 8 * slot);
    }
    drain();
    named_sync(1, 32 * kConsumers);
    if (aborted || *s_abort) break;
    // ---- epilogue: dequantize and store this item's outputs, clear s_acc
    auto store_out = [&](int e, float as, float ws) {
      const int mm = e / R, rr = e - mm * R;
      const int v = s_acc[e];
      s_acc[e] = 0;
      if (rr < f.ntiles * 16) {
        const int m = 16 * f.z + mm, n = f.r0 + rr;
        const size_t o = (size_t)m * p.N + n;
        const float yv = __fmul_rn(__fmul_rn((float)v, as), ws);
        if (p.out_dtype == 0) {
          reinterpret_cast<float*>(p.y)[o] = yv;
        } else {
          __nv_bfloat16* yb = reinterpret_cast<__nv_bfloat16*>(p.y) + o;
          // out_dtype 2: residual add into the bf16 output, y = bf16(y + result)
          *yb = __float2bfloat16_rn(p.out_dtype == 2 ? __fadd_rn(__bfloat162float(*yb), yv) : yv);
        }
        if (p.acc_debug) p.acc_debug[o] = v;
      }
    };
#pragma unroll
    for (int j = 0; j < NPF; ++j) {
      const int e = (int)threadIdx.x - 32 + j * 32 * kConsumers;
      if (e < nout) store_out(e, pf_as[j], pf_ws[j]);
    }
    for (int e = (int)threadIdx.x - 32 + NPF * 32 * kConsumers; e < nout; e += 32 * kConsumers) {
      const int mm = e / R, rr = e - mm * R;
      store_out(e, rr < f.ntiles * 16 ? __ldg(p.act_scale + 16 * f.z + mm) : 0.0f,
                rr < f.ntiles * 16 ? __ldg(p.w_scale + f.r0 + rr) : 0.0f);
    }
    named_sync(1, 32 * kConsumers);
  }
}

// x_q -> activation operands, for callers that did not get them from quant_act.
__global__ void act_ops_from_codes_kernel(const int8_t* __restrict__ x_q, int64_t M, int64_t K,
                                          int64_t Kp, uint8_t* __restrict__ ops) {
  pdl_wait();
  pdl_launch_dependents();
  const int64_t per_row = Kp >> 4;
  for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < M * per_row;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int64_t m = idx / per_row, k = (idx - m * per_row) << 4;
    int q[16];
#pragma unroll
    for (int hv = 0; hv < 2; ++hv) {
      if (k + 8 * hv < K) {
        const uint2 v = *reinterpret_cast<const uint2*>(x_q + m * K + k + 8 * hv);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          q[8 * hv + j] = (int)(int8_t)(v.x >> (8 * j));
          q[8 * hv + j + 4] = (int)(int8_t)(v.y >> (8 * j));
        }
      } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) q[8 * hv + j] = 0;
      }
    }
    write_act_ops16_any(ops, M, m, k, Kp, q);
  }
}

// Segments per stage: a divisor of nseg (no half-empty last stage) with two
// units per segment = one unit per consumer warp.
int stage_segments(int nseg, int max_sbk) {
  int best = 0;
  for (int d = 1; d <= max_sbk && d <= nseg; ++d)
    if (nseg % d == 0) best = d;
  if (best >= 3 || best == nseg) return best;
  return nseg < max_sbk ? nseg : max_sbk;            // few divisors: accept a partial last stage
}

template <int T, int MT, int CMAX>
cudaError_t launch_t(DecodeParams& p, int sms, bool pdl, cudaStream_t stream) {
  constexpr int R = T * 16;
  const int Mz_max = p.M < 16 ? p.M : 16;
  const int64_t Kp = (int64_t)p.nseg * 512;
  // With one token tile and operands of at most 112 KB, the operands are copied
  // once and stay resident; stages then carry weights only (~32 KB each).
  const int64_t bres_need = 2 * (int64_t)Mz_max * Kp;
  const bool resident = p.ztiles == 1 && bres_need <= 112 * 1024;
  p.bres_bytes = resident ? (int)bres_need : 0;
  int SBK;
  if (resident) {
    SBK = stage_segments(p.nseg, 16 / T > 1 ? 16 / T : 1);
  } else {
    // largest stage that leaves room for two of them in shared memory
    SBK = stage_segments(p.nseg, CMAX / 2);
    while (SBK > 1 && 2L * (T * SBK * 2048 + SBK * 1024 * Mz_max) + 16 * R * 4 + 1024 > 210L * 1024)
      SBK = stage_segments(p.nseg, SBK - 1);
  }
  // consumers: one or more whole units each (a unit = 256 k of a segment)
  int C = 2 * SBK;
  while (C > CMAX) {
    int d = CMAX;
    while (d > 1 && (2 * SBK) % d != 0) --d;
    C = d >= 2 ? d : CMAX;
    break;
  }
  p.SBK = SBK;
  p.stage_w_bytes = T * SBK * 2048;
  p.stage_bytes = p.stage_w_bytes + (resident ? 0 : SBK * 1024 * Mz_max);
  int NS = (int)((200L * 1024 - p.bres_bytes - 16 * R * 4) / p.stage_bytes);
  if (NS < 2) NS = 2;
  if (NS > kMaxStages) NS = kMaxStages;
  p.NS = NS;
  const size_t smem = 128 + (size_t)NS * p.stage_bytes + p.bres_bytes + 16 * R * 4 + (2 * kMaxStages + 1) * 8 + 16;
  if (smem > 220 * 1024) return cudaErrorInvalidValue;
  static bool attr_set = false;   // per template instance
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(decode_mma_kernel<T, MT, CMAX>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, 220 * 1024);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  cudaLaunchConfig_t cfg = {};
  const int grid = p.items < sms ? p.items : sms;
  cfg.gridDim = dim3((unsigned)grid, 1, 1);
  cfg.blockDim = dim3(32 * (1 + C), 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  cudaError_t e = cudaLaunchKernelEx(&cfg, decode_mma_kernel<T, MT, CMAX>, p);
  count_launches(1);
  return e;
}

}  // namespace

size_t act_ops_bytes(int64_t M, int64_t K) {
  return (size_t)(2 * (act_ops_prefill(M) ? act_ops_mpad(M) : M) * act_ops_kpad(K));
}

cudaError_t launch_act_ops_from_codes(const int8_t* x_q, int64_t M, int64_t K, uint8_t* ops,
                                      bool pdl, cudaStream_t stream) {
  const int64_t Kp = act_ops_kpad(K);
  const int64_t work = M * (Kp >> 4);
  int64_t blocks = (work + 255) / 256;
  if (blocks > (int64_t)num_sms() * 8) blocks = (int64_t)num_sms() * 8;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks, 1, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  cudaError_t e = cudaLaunchKernelEx(&cfg, act_ops_from_codes_kernel, x_q, M, K, Kp, ops);
  count_launches(1);
  return e;
}

cudaError_t launch_decode_mma(const uint8_t* x_ops, const float* act_scale, const uint8_t* packed,
                              const float* w_scale, int64_t M, int64_t N, int64_t K, int out_dtype,
                              void* y, int32_t* acc_debug, int* dev_err, bool pdl,
                              cudaStream_t stream) {
  const int sms = num_sms();
  DecodeParams p = {};
  p.packed = packed;
  p.x_ops = x_ops;
  p.act_scale = act_scale;
  p.w_scale = w_scale;
  p.y = y;
  p.acc_debug = acc_debug;
  p.dev_err = dev_err;
  p.M = (int)M;
  p.N = (int)N;
  p.K = (int)K;
  p.out_dtype = out_dtype;
  p.ztiles = (int)((M + 15) / 16);
  p.nseg = (int)(act_ops_kpad(K) / 512);
  const int64_t tiles = N / 16;
  // T row tiles per item.  Measured on the decode shapes (N = 2560 .. 28672,
  // M = 1 .. 16): T = 2 beats T = 1 (more per-item synchronisation and epilogue
  // work per weight byte) and T = 4 (fewer items than SMs on small N).
  const int T = tiles >= 2 ? 2 : 1;
  p.groups = (int)((tiles + T - 1) / T);
  const int64_t items = (int64_t)p.groups * p.ztiles;
  if (items > (1LL << 30)) return cudaErrorInvalidValue;
  p.items = (int)items;
  const bool two = M > 8;
  if (T == 2)
    return two ? launch_t<2, 2, 8>(p, sms, pdl, stream) : launch_t<2, 1, 14>(p, sms, pdl, stream);
  return two ? launch_t<1, 2, 8>(p, sms, pdl, stream) : launch_t<1, 1, 14>(p, sms, pdl, stream);
}

}  // namespace bitlinear
