#!/usr/bin/env python
"""Benchmark of the BitNet b1.58 BitLinear forward on B300.

Headline workload: decode through the BitLinear projections of a 2B-class
BitNet b1.58 (hidden 2560, FFN 6912; QKV 2560->3840, O 2560->2560, gate+up
2560->2x6912, down 6912->2560) at M = 1 and M = 8 tokens, over 30 layers of
distinct weights (520 MB of packed weights per pass, more than 4x the 126 MB
L2, so no pass is served from L2).  One step = for M in (1, 8): for each layer
and projection: the BitLinear layer through the one-call API
bitlinear_linear_forward (RMSNorm + int8 quantization of the input, the ternary
contraction with fused dequantization; one kernel at M = 1, two at M = 8).
Weights are packed once before timing (offline step).

Metric: packed-weight GB/s (packed bytes streamed per step / step time).  The
same line carries "prefill": the M = 2048 prefill of the 8B-class shapes
(4096->14336, 14336->4096) in int8-equivalent TOPS (2 M N K / time).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload decode_2b|stack_2b]

--workload stack_2b times bitlinear_block_forward over the 30-layer linear stack
of the 2B-class model (hidden 2560, QKV 3840, FFN 6912, ReLU^2 gating) at
M = 1, 8 (decode) and 512 (prefill) tokens.

N > 1 runs N independent replicas (one per GPU, launched by torchrun); value is
the aggregate over ranks and the step time the max over ranks.  The reference
arm times the CPU oracle (the plain single-threaded C definition) on a bounded
sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "BitLinear decode packed-weight GB/s vs HBM peak; M=2048 prefill int8 TOPS"
WORKLOAD = "decode_2b"
LAYERS = 30
RMS_EPS = 1e-5


def log(*a):
    print(*a, file=sys.stderr, flush=True)


# ---------------------------------------------------------------------------
# environment helpers
# ---------------------------------------------------------------------------

def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")),
            int(os.environ.get("WORLD_SIZE", "1")))


def max_over_ranks(value: float, pg, device) -> float:
    """The largest `value` over all ranks (the slowest replica sets the step time);
    `pg` is torch.distributed (or None for one process)."""
    if pg is None:
        return float(value)
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def aggregate_gbs(world: int, bytes_per_step_per_rank: int, ms_per_step: float) -> float:
    """Whole-job GB/s of N replicas that each stream `bytes_per_step_per_rank` per step,
    timed by the slowest one."""
    return world * bytes_per_step_per_rank / (ms_per_step * 1e-3) / 1e9


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    except Exception:
        return 6400.0, 1800.0, "fallback"


class ClockSampler:
    """Samples SM clock and clock-event reasons while the timed region runs: NVML
    (pynvml) polled every ~2 ms when importable, else `nvidia-smi -lms 50`."""
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown", 0x2: "applications_clocks",
               0x100: "display_clock", 0x10: "sync_boost"}

    def __init__(self, index: int):
        self.index = index
        self.samples, self.reasons, self.names, self.mode = [], 0, set(), None
        self.max_mhz = None
        self._stop = threading.Event()
        try:
            import pynvml
            pynvml.nvmlInit()
            self.nv = pynvml
            self.h = pynvml.nvmlDeviceGetHandleByIndex(index)
            self.max_mhz = float(pynvml.nvmlDeviceGetMaxClockInfo(self.h, pynvml.NVML_CLOCK_SM))
            self.mode = "nvml"
        except Exception:
            self.mode = "smi"

    def _sample(self):
        nv = self.nv
        self.samples.append(float(nv.nvmlDeviceGetClockInfo(self.h, nv.NVML_CLOCK_SM)))
        self.reasons |= nv.nvmlDeviceGetCurrentClocksEventReasons(self.h)

    def _run(self):
        while not self._stop.is_set():
            self._sample()
            time.sleep(0.002)

    def __enter__(self):
        if self.mode == "nvml":
            self._sample()
            self._t = threading.Thread(target=self._run, daemon=True)
            self._t.start()
        else:
            import subprocess
            import tempfile
            self._f = tempfile.TemporaryFile(mode="w+")
            q = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
                 "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
                 "clocks_event_reasons.sw_power_cap")
            try:
                self._p = subprocess.Popen(["nvidia-smi", f"--query-gpu={q}", "--format=csv,noheader,nounits",
                                            "-i", str(self.index), "-lms", "50"], stdout=self._f,
                                           stderr=subprocess.DEVNULL)
                time.sleep(0.3)
            except Exception:
                self._p = None
        return self

    def __exit__(self, *exc):
        if self.mode == "nvml":
            self._stop.set()
            self._t.join()
            self._sample()
        elif self._p is not None:
            time.sleep(0.1)
            self._p.terminate()
            self._p.wait()
            self._f.seek(0)
            labels = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
            for line in self._f.read().splitlines():
                f = [x.strip() for x in line.split(",")]
                if len(f) < 6:
                    continue
                try:
                    self.samples.append(float(f[0]))
                    self.max_mhz = float(f[1])
                except ValueError:
                    continue
                for lab, v in zip(labels, f[2:6]):
                    if v.lower() == "active":
                        self.names.add(lab)

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": [], "samples": 0,
                    "source": self.mode}
        names = set(self.names) | {n for b, n in self.REASONS.items() if self.reasons & b}
        return {"sm_mhz": float(statistics.median(self.samples)), "sm_max_mhz": self.max_mhz,
                "reasons": sorted(names), "samples": len(self.samples), "source": self.mode}


# ---------------------------------------------------------------------------
# CPU baseline: the oracle, as it stands, on a bounded sample
# ---------------------------------------------------------------------------

_ORACLE_SAMPLE = None


def _oracle_inputs():
    """Layer 0 of the decode workload, ternarized by the oracle (offline step, not timed)."""
    global _ORACLE_SAMPLE
    if _ORACLE_SAMPLE is None:
        import oracle
        from bitlinear_rmsnorm_token_int8_b300 import synth
        wl = synth.WORKLOADS[WORKLOAD]
        mats = []
        for pi, p in enumerate(wl.projections):
            W = synth.latent_weights(p.N, p.K, synth.weight_seed(wl.seed, 0, pi)).numpy()
            _, gamma, wq = oracle.pack_weights(W)
            mats.append((p, gamma, wq))
        xs = {}
        for M in wl.tokens:
            for K in sorted({p.K for p in wl.projections}):
                xs[(M, K)] = (synth.bf16_bits(synth.activations(M, K, synth.act_seed(wl.seed, M, K), outliers=False)),
                              synth.bf16_bits(synth.rms_gains(K, synth.gain_seed(wl.seed, 0, K))))
        _ORACLE_SAMPLE = (wl, mats, xs)
    return _ORACLE_SAMPLE


def oracle_sample(seconds: float = 12.0):
    """Times the CPU oracle as it stands (act-quant + add/skip/subtract contraction +
    dequant) on layer 0 of the decode workload at M = 1 and M = 8, whole passes
    repeated until ~`seconds` have passed.  Returns (packed-weight GB/s, seconds, passes)."""
    import oracle
    wl, mats, xs = _oracle_inputs()
    done_bytes, t0, reps = 0, time.perf_counter(), 0
    while True:
        for M in wl.tokens:
            for p, gamma, wq in mats:
                xb, gb = xs[(M, p.K)]
                xq, sig = oracle.act_quant(xb, gb, RMS_EPS)
                acc = oracle.ternary_matmul(xq, wq)
                oracle.dequant(acc, sig, np.full(p.N, float(gamma)))
                done_bytes += p.N * p.K // 4
        reps += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    return done_bytes / el / 1e9, el, reps


def reference_arm(args):
    rank, _, world = dist_env()
    if rank != 0:
        return 0
    import oracle
    oracle.build()
    _oracle_inputs()
    per_step = min(args.ref_seconds, 150.0 / max(args.steps, 1))   # whole arm within a few minutes
    t0 = time.perf_counter()
    gbs_list = []
    for _ in range(args.steps):
        gbs, _, _ = oracle_sample(per_step)
        gbs_list.append(gbs)
    el = time.perf_counter() - t0
    value = float(statistics.mean(gbs_list))
    sample = (f"layer 0 of {LAYERS} (QKV, O, gate+up, down) at M=1 and M=8 per step, "
              f"~{per_step:.1f} s per step, single-threaded C oracle")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int32",
        "data": "synthetic", "config": {"workload": WORKLOAD, "layers_sampled": 1, "tokens": [1, 8]},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

def traffic_record(kernel_srcs):
    """ncu DRAM bytes per launch recorded for the current sources of the kernels, or None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        rec = json.load(open(path))
    except Exception:
        return None
    h = hashlib.sha256()
    for src in kernel_srcs:
        h.update(open(src, "rb").read())
    sha = h.hexdigest()[:16]
    r = rec.get(WORKLOAD)
    if not r or r.get("source_sha") != sha:
        return None
    return float(r["dram_bytes_per_launch"])


def measure_prefill(bl, synth, torch, dev, steps, warmup):
    """M = 2048 prefill of the 8B-class shapes (4096->14336, 14336->4096): per shape one
    graph of the whole BitLinear layer (bitlinear_linear_forward: RMSNorm + quantization
    into the operand form, then the contraction); CUDA events around `steps` replays.
    Reports int8-equivalent TOPS (2 M N K / time) of the quant + contraction pair and
    of the contraction alone, and the contraction's tensor-core rate against the
    measured peak: it issues two e4m3 MMAs per int8 product, i.e. 4 M N K fp8 FLOP."""
    wl = synth.WORKLOADS["prefill_8b_m2048"]
    M = wl.tokens[0]
    stream = torch.cuda.Stream(device=dev)
    out = {"workload": "prefill_8b_m2048", "tokens": M, "shapes": []}
    tot_ops = tot_ms = tot_fwd_ms = 0.0
    for pi, p in enumerate(wl.projections):
        W = synth.latent_weights_device(p.N, p.K, synth.weight_seed(wl.seed, 0, pi), dev)
        packed, w_scale, _ = bl.bitlinear_pack_weights(W)
        del W
        x = synth.activations(M, p.K, synth.act_seed(wl.seed, M, p.K), outliers=True).to(dev)
        g = synth.rms_gains(p.K, synth.gain_seed(wl.seed, 0, pi)).to(dev)
        sc = torch.empty(M + 4, dtype=torch.float32, device=dev)[:M]
        ops = torch.empty(bl.bitlinear_act_ops_bytes(M, p.K), dtype=torch.uint8, device=dev)
        ws = torch.empty(bl.bitlinear_linear_workspace_bytes(M, p.N, p.K), dtype=torch.uint8, device=dev)
        y = torch.empty((M, p.N), dtype=torch.bfloat16, device=dev)
        # operands and scales for the contraction-only graph
        bl.bitlinear_quant_act(x, g, RMS_EPS, act_scale=sc, x_ops=ops)
        graphs = {}
        with torch.cuda.stream(stream):
            for kind in ("pair", "fwd"):
                def run(kind=kind):
                    if kind == "pair":
                        bl.bitlinear_linear_forward(x, g, RMS_EPS, packed, w_scale, out_dtype=torch.bfloat16, y=y,
                                                    workspace=ws, flags=bl.FLAG_PDL, stream=stream)
                    else:
                        bl.bitlinear_forward(None, sc, packed, w_scale, out_dtype=torch.bfloat16, y=y, x_ops=ops,
                                             flags=bl.FLAG_PDL, K=p.K, stream=stream)
                run()
                stream.synchronize()
                gr = torch.cuda.CUDAGraph()
                with torch.cuda.graph(gr, stream=stream):
                    run()
                graphs[kind] = gr
            ms = {}
            for kind, gr in graphs.items():
                for _ in range(max(warmup, 3)):
                    gr.replay()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                for _ in range(steps):
                    gr.replay()
                e1.record(stream)
                stream.synchronize()
                ms[kind] = e0.elapsed_time(e1) / steps
        ops_ = 2.0 * M * p.N * p.K
        out["shapes"].append({"K": p.K, "N": p.N, "ms": ms["pair"], "fwd_ms": ms["fwd"],
                              "int8_equiv_tops": ops_ / (ms["pair"] * 1e9),
                              "fwd_int8_equiv_tops": ops_ / (ms["fwd"] * 1e9)})
        tot_ops += ops_
        tot_ms += ms["pair"]
        tot_fwd_ms += ms["fwd"]
        del packed, w_scale, x, ops, ws, y, graphs
    _, bf16_tf, src = measured_peaks()
    fp8_peak = 2.0 * bf16_tf          # e4m3 dense rate = 2x bf16 (nominal ratio)
    fwd_tflops = 2.0 * tot_ops / (tot_fwd_ms * 1e9)
    out.update({"int8_equiv_tops": tot_ops / (tot_ms * 1e9), "fwd_int8_equiv_tops": tot_ops / (tot_fwd_ms * 1e9),
                "roofline": {"bound": "tensor", "achieved": fwd_tflops, "unit": "TFLOP/s (e4m3 MMA)",
                             "peak": fp8_peak, "frac": fwd_tflops / fp8_peak,
                             "peak_source": f"{src} bf16 cuBLAS x 2 (nominal e4m3:bf16 ratio)"}})
    return out


def our_arm(args):
    import torch
    import bitlinear_rmsnorm_token_int8_b300 as bl
    from bitlinear_rmsnorm_token_int8_b300 import synth

    rank, local_rank, world = dist_env()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist
    bl.lib()
    wl = synth.WORKLOADS[WORKLOAD]
    layers = args.layers

    # ---- weights (offline step, not timed)
    weights = []
    for layer in range(layers):
        row = []
        for pi, p in enumerate(wl.projections):
            W = synth.latent_weights_device(p.N, p.K, synth.weight_seed(wl.seed, layer, pi) + 7919 * rank, dev)
            packed, w_scale, _ = bl.bitlinear_pack_weights(W)
            del W
            row.append((p, packed, w_scale))
        weights.append(row)
    torch.cuda.synchronize()
    assert bl.bitlinear_get_device_error() == 0

    # ---- activations and buffers
    Ks = sorted({p.K for p in wl.projections})
    xs, gains, xq, sc, ops, ys, lws = {}, {}, {}, {}, {}, {}, {}
    for K in Ks:
        gains[K] = synth.rms_gains(K, synth.gain_seed(wl.seed, 0, K)).to(dev)
    for M in wl.tokens:
        for K in Ks:
            xs[(M, K)] = synth.activations(M, K, synth.act_seed(wl.seed, M, K), outliers=False).to(dev)
            xq[(M, K)] = torch.empty((M, K), dtype=torch.int8, device=dev)
            sc[(M, K)] = torch.empty(M + 4, dtype=torch.float32, device=dev)[:M]
            ops[(M, K)] = torch.empty(bl.bitlinear_act_ops_bytes(M, K), dtype=torch.uint8, device=dev)
        for p in wl.projections:
            ys[(M, p.N)] = torch.empty((M, p.N), dtype=torch.bfloat16, device=dev)
            lws[(M, p.N, p.K)] = torch.empty(max(16, bl.bitlinear_linear_workspace_bytes(M, p.N, p.K)),
                                             dtype=torch.uint8, device=dev)

    packed_bytes_step = sum(p.N * p.K // 4 for _ in wl.tokens for row in weights for (p, _, _) in row)

    stream = torch.cuda.Stream(device=dev)
    FL = bl.FLAG_PDL

    def route(M, p):
        return bl.bitlinear_linear_route(M, p.N, p.K)

    def alg_bytes(M, p):
        # per launch of the kernel timed for the roofline: packed weights, its activation
        # input (bf16 x and gain for the one-token layer kernel, int8 codes for the code
        # kernel, two e4m3 planes for tcgen05), scales, bf16 outputs
        r = route(M, p)
        acts = (2 * M * p.K + 2 * p.K if r == bl.ROUTE_FUSED else M * p.K if r == bl.ROUTE_CODES
                else 2 * M * p.K)
        return p.N * p.K // 4 + acts + 4 * M + 4 * p.N + 2 * M * p.N

    def layer(M, x, p, packed, w_scale, y):
        # one BitLinear layer through the public one-call API (RMSNorm + quantization +
        # contraction): one kernel for one token, quantization + contraction otherwise
        bl.bitlinear_linear_forward(x, gains[p.K], RMS_EPS, packed, w_scale, out_dtype=torch.bfloat16, y=y,
                                    workspace=lws[(M, p.N, p.K)], flags=FL, stream=stream)

    def step():
        """One pass: for M in (1, 8), for every layer and projection, the BitLinear layer
        (bitlinear_linear_forward: RMSNorm, int8 quantization and the contraction)."""
        for M in wl.tokens:
            for row in weights:
                for (p, packed, w_scale) in row:
                    layer(M, xs[(M, p.K)], p, packed, w_scale, ys[(M, p.N)])

    def barrier():
        if pg is not None:
            pg.barrier()

    # ---- the step as one CUDA graph (kernels chained by programmatic dependent launch)
    with torch.cuda.stream(stream):
        step()                                   # eager warm-up (module load, first launches)
        stream.synchronize()
        graph = torch.cuda.CUDAGraph()
        l0 = bl.bitlinear_kernel_launches()
        with torch.cuda.graph(graph, stream=stream):
            step()
        launches_per_step = bl.bitlinear_kernel_launches() - l0
    torch.cuda.synchronize()

    # ---- warmup: W replays, then more until ~1 s has passed (clock ramp-up)
    t0 = time.perf_counter()
    n = 0
    while n < args.warmup or time.perf_counter() - t0 < 1.0:
        graph.replay()
        n += 1
        if n % 20 == 0:
            torch.cuda.synchronize()
    torch.cuda.synchronize()

    # ---- timed region: K replays of the step
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    with ClockSampler(local_rank) as clk:
        with torch.cuda.stream(stream):
            start.record(stream)
            for s in range(args.steps):
                graph.replay()
            end.record(stream)
        torch.cuda.synchronize()
    barrier()
    launches = launches_per_step * args.steps
    ms = max_over_ranks(start.elapsed_time(end) / args.steps, pg, dev)
    value = aggregate_gbs(world, packed_bytes_step, ms)

    # ---- per-launch durations of the contraction kernel (for one token the layer kernel,
    #      which also quantizes).  For each (M, projection) a CUDA graph holds the 30
    #      layers' launches back to back (distinct weights, chained by programmatic
    #      dependent launch as in the step); CUDA events on the launching stream bracket K
    #      replays, so the average is the kernel's duration in a stream of launches, not
    #      host launch latency.  Codes, scales and operand planes for the contraction-only
    #      launches come from one quantization per (M, K) beforehand.
    with torch.cuda.stream(stream):
        for M in wl.tokens:
            for K in Ks:
                bl.bitlinear_quant_act(xs[(M, K)], gains[K], RMS_EPS, x_q=xq[(M, K)], act_scale=sc[(M, K)],
                                       x_ops=ops[(M, K)], stream=stream)
    fwd_graphs = []
    with torch.cuda.stream(stream):
        for M in wl.tokens:
            for pi, p in enumerate(wl.projections):
                def fwd_only(M=M, pi=pi, p=p):
                    for row in weights:
                        _, packed, w_scale = row[pi]
                        if route(M, p) == bl.ROUTE_FUSED:    # the layer is one kernel
                            layer(M, xs[(M, p.K)], p, packed, w_scale, ys[(M, p.N)])
                        else:                                  # the contraction kernel alone
                            codes = route(M, p) == bl.ROUTE_CODES
                            bl.bitlinear_forward(xq[(M, p.K)] if codes else None, sc[(M, p.K)], packed, w_scale,
                                                 out_dtype=torch.bfloat16, y=ys[(M, p.N)],
                                                 x_ops=None if codes else ops[(M, p.K)], K=p.K, flags=FL,
                                                 stream=stream)
                fwd_only()
                stream.synchronize()
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream):
                    fwd_only()
                fwd_graphs.append((M, p, g))
        for _, _, g in fwd_graphs:
            g.replay()
        stream.synchronize()
        fwd_ms = []            # per-launch ms, one entry per forward launch of a step
        per_shape = []         # per (M, projection): launch time and algorithmic GB/s
        for M, p, g in fwd_graphs:
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(args.steps):
                g.replay()
            e1.record(stream)
            stream.synchronize()
            per_launch = e0.elapsed_time(e1) / (args.steps * len(weights))
            fwd_ms.extend([per_launch] * len(weights))
            alg = alg_bytes(M, p)
            per_shape.append({"tokens": M, "projection": p.name, "launch_us": per_launch * 1e3,
                              "alg_gbs": alg / (per_launch * 1e-3) / 1e9})
    alg_bytes_fwd = []
    for M, p, _ in fwd_graphs:
        for _ in weights:
            alg_bytes_fwd.append(alg_bytes(M, p))
    per_step_launches = len(alg_bytes_fwd)

    # ---- end to end through the public API: pinned host inputs in, bf16 outputs out.
    #      Every projection of the step gets its own input rows; they travel to the
    #      device as one copy from one pinned buffer, and all outputs come back as one
    #      copy, the way a caller stages a step's data.
    in_off, out_off = {}, {}
    h2d = d2h = 0
    for M in wl.tokens:
        for li, row in enumerate(weights):
            for pi, (p, _, _) in enumerate(row):
                in_off[(M, li, pi)] = h2d // 2
                out_off[(M, li, pi)] = d2h // 2
                h2d += M * p.K * 2
                d2h += M * p.N * 2
    host_in = torch.empty(h2d // 2, dtype=torch.bfloat16, pin_memory=True)
    host_out = torch.empty(d2h // 2, dtype=torch.bfloat16, pin_memory=True)
    for M in wl.tokens:
        for li, row in enumerate(weights):
            for pi, (p, _, _) in enumerate(row):
                o = in_off[(M, li, pi)]
                host_in[o:o + M * p.K].copy_(xs[(M, p.K)].reshape(-1).cpu())
    dev_in = torch.empty_like(host_in, device=dev)
    dev_out = torch.empty_like(host_out, device=dev)

    side = torch.cuda.Stream(device=dev)       # host<->device copies, beside the kernels
    in_rng = {}                                 # element range of each pass's inputs
    for M in wl.tokens:
        lo = in_off[(M, 0, 0)]
        last = (M, len(weights) - 1, len(wl.projections) - 1)
        in_rng[M] = (lo, in_off[last] + M * wl.projections[-1].K)
    out_rng = {}                                # element range of each (pass, layer)'s outputs
    for M in wl.tokens:
        for li in range(len(weights)):
            lo = out_off[(M, li, 0)]
            out_rng[(M, li)] = (lo, out_off[(M, li, len(wl.projections) - 1)] + M * wl.projections[-1].N)

    def e2e_step():
        """Inputs in, per projection RMSNorm + quant and the contraction, outputs out.  The
        copies run on a side stream: each pass's inputs as one copy (the second pass's
        while the first computes), each layer's outputs as soon as the layer is done."""
        side.wait_stream(stream)
        ev_in = {}
        with torch.cuda.stream(side):
            for M in wl.tokens:
                lo, hi = in_rng[M]
                dev_in[lo:hi].copy_(host_in[lo:hi], non_blocking=True)
                ev_in[M] = torch.cuda.Event()
                ev_in[M].record(side)
        for M in wl.tokens:
            stream.wait_event(ev_in[M])
            for li, row in enumerate(weights):
                for pi, (p, packed, w_scale) in enumerate(row):
                    o = in_off[(M, li, pi)]
                    x = dev_in[o:o + M * p.K].view(M, p.K)
                    yo = out_off[(M, li, pi)]
                    y = dev_out[yo:yo + M * p.N].view(M, p.N)
                    layer(M, x, p, packed, w_scale, y)
                done = torch.cuda.Event()
                done.record(stream)
                side.wait_event(done)
                with torch.cuda.stream(side):
                    lo, hi = out_rng[(M, li)]
                    host_out[lo:hi].copy_(dev_out[lo:hi], non_blocking=True)
        stream.wait_stream(side)

    # the e2e step as one graph too: copy nodes from/to pinned host memory around the
    # library calls, so the number is not Python launch overhead
    with torch.cuda.stream(stream):
        e2e_step()
        stream.synchronize()
        e2e_graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(e2e_graph, stream=stream):
            e2e_step()
        for _ in range(max(args.warmup, 1)):
            e2e_graph.replay()
        torch.cuda.synchronize()
        barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            e2e_graph.replay()
        e1.record(stream)
        torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, pg, dev)
    e2e_value = aggregate_gbs(world, packed_bytes_step, e2e_ms)

    # ---- roofline of the dominant kernel (the contraction)
    hbm, bf16_tf, peak_src = measured_peaks()
    achieved = sum(alg_bytes_fwd) / (sum(fwd_ms) * 1e-3) / 1e9
    csrc = os.path.join(ROOT, "bitlinear_rmsnorm_token_int8_b300", "csrc")
    traffic = traffic_record([os.path.join(csrc, "decode_dp4a.cu"), os.path.join(csrc, "quant_math.cuh"),
                              os.path.join(csrc, "decode_tc.cu")])
    roofline = {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                "traffic": traffic, "peak_source": peak_src,
                "kernel": "the decode contraction + dequant of each projection: at M = 1 linear_dp4a_kernel "
                          "(the whole layer: RMSNorm, quantization, int8-code contraction, CUDA cores), at "
                          "M = 8 decode_tc_kernel (tcgen05)",
                "timing": "CUDA events around K replays of a graph of the 30 layers' launches per (M, projection)",
                "alg_bytes_per_launch": sum(alg_bytes_fwd) / len(alg_bytes_fwd),
                "avg_launch_us": sum(fwd_ms) / len(fwd_ms) * 1e3,
                "share_of_step": sum(fwd_ms) / ms if ms > 0 else None,
                "per_shape": per_shape}

    # ---- CPU baseline (rank 0, N = 1 only)
    prefill = None
    if not args.no_prefill:
        prefill = measure_prefill(bl, synth, torch, dev, max(3, args.steps), args.warmup)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        gbs, el, reps = oracle_sample(args.ref_seconds)
        cpu = {"value": gbs, "unit": "GB/s", "cores": 1, "kind": "oracle",
               "sample": f"layer 0 of {LAYERS} (QKV, O, gate+up, down) at M=1 and M=8, {reps} passes in {el:.1f} s"}

    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "int32",
        "data": "synthetic (seeded N(0,0.02) latent weights, N(0,1) bf16 activations)",
        "config": {"workload": WORKLOAD, "layers": layers, "tokens": list(wl.tokens),
                   "projections": [[p.name, p.K, p.N] for p in wl.projections],
                   "packed_bytes_per_step": packed_bytes_step,
                   "l2": "no flush: 520 MB of distinct packed weights per pass (> 4x the 126 MB L2)",
                   "launch": "one CUDA graph per step; kernels chained by programmatic dependent launch",
                   "parallelism": f"replicas x{world}"},
        "e2e": {"value": e2e_value, "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": int(launches),
        "roofline": roofline,
        "cpu_baseline": cpu,
        "clocks": clk.summary(),
        "prefill": prefill,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if pg is not None:
        pg.destroy_process_group()
    return 0


def stack_arm(args):
    """30-layer BitLinear stack (bitlinear_block_forward) at M = 1, 8 and 512 tokens."""
    import torch
    import bitlinear_rmsnorm_token_int8_b300 as bl
    from bitlinear_rmsnorm_token_int8_b300 import synth

    rank, local_rank, world = dist_env()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    wl = synth.WORKLOADS["stack_2b"]
    H, NQKV, F = 2560, 3840, 6912
    layers, packed_bytes = [], 0
    for l in range(args.layers):
        layer = {}
        for j, (name, shapes) in enumerate({"qkv": [(NQKV, H)], "o": [(H, H)], "gate_up": [(F, H), (F, H)],
                                            "down": [(H, F)]}.items()):
            Ws = [synth.latent_weights_device(n, k, synth.weight_seed(wl.seed, l, 3 * j + i) + 7919 * rank, dev)
                  for i, (n, k) in enumerate(shapes)]
            layer[name], layer[name + "_scale"] = bl.pack_stacked(Ws)
            packed_bytes += sum(n * k // 4 for n, k in shapes)
            del Ws
        for j, (name, k) in enumerate({"gain_qkv": H, "gain_o": H, "gain_gate_up": H, "gain_down": F}.items()):
            layer[name] = synth.rms_gains(k, synth.gain_seed(wl.seed, l, j)).to(dev)
        layers.append(layer)
    torch.cuda.synchronize()
    stream = torch.cuda.Stream(device=dev)
    results = {}
    for M in wl.tokens:
        x0 = synth.activations(M, H, synth.act_seed(wl.seed, M, H), outliers=True).to(dev)
        x = x0.clone()
        ws = torch.empty(bl.bitlinear_block_workspace_bytes(M, H, NQKV, F) + 256, dtype=torch.uint8, device=dev)
        with torch.cuda.stream(stream):
            bl.bitlinear_block_forward(layers, x, H, NQKV, F, RMS_EPS, workspace=ws, flags=bl.FLAG_PDL, stream=stream)
            stream.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                bl.bitlinear_block_forward(layers, x, H, NQKV, F, RMS_EPS, workspace=ws, flags=bl.FLAG_PDL,
                                           stream=stream)
            for _ in range(max(args.warmup, 3)):
                g.replay()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(args.steps):
                g.replay()
            e1.record(stream)
            stream.synchronize()
        assert bl.bitlinear_get_device_error(stream) == 0
        ms = e0.elapsed_time(e1) / args.steps
        results[M] = {"ms_per_forward": ms, "tokens_per_s": M / (ms * 1e-3),
                      "packed_gbs": packed_bytes / (ms * 1e-3) / 1e9,
                      "int8_equiv_tops": 2.0 * M * 4 * packed_bytes / (ms * 1e9)}
    line = {"metric": METRIC, "value": results[wl.tokens[0]]["packed_gbs"], "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": results[wl.tokens[0]]["ms_per_forward"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int32",
            "data": "synthetic", "config": {"workload": "stack_2b", "layers": args.layers, "hidden": H,
                                            "qkv": NQKV, "ffn": F, "packed_bytes_per_forward": packed_bytes},
            "per_tokens": {str(k): v for k, v in results.items()}}
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--layers", type=int, default=LAYERS)
    ap.add_argument("--ref-seconds", type=float, default=12.0, help="CPU oracle seconds per sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-prefill", action="store_true", help="skip the M=2048 prefill measurement")
    ap.add_argument("--workload", choices=["decode_2b", "stack_2b"], default="decode_2b")
    args = ap.parse_args()
    if args.impl == "reference":
        return reference_arm(args)
    if args.workload == "stack_2b":
        return stack_arm(args)
    return our_arm(args)


if __name__ == "__main__":
    sys.exit(main())
