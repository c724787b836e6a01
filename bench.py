#!/usr/bin/env python
"""Benchmark of the BitNet b1.58 BitLinear forward on one B300.

Headline workload (decode_8b): decode through the BitLinear projections of an
8B-class BitNet b1.58 (hidden 4096, FFN 14336; QKV 4096->6144, O 4096->4096,
gate+up 4096->2x14336, down 14336->4096) at M = 1, 4 and 16 tokens, over 32
layers of distinct weights (1.74 GB of packed weights per pass, 14x the 126 MB
L2, so no pass is served from L2).  One step = for M in (1, 4, 16): for each
layer and projection: the BitLinear layer through the one-call API
bitlinear_linear_forward (RMSNorm + int8 quantization of the input, the ternary
contraction with fused dequantization; one kernel for one token with K <= 8192,
two otherwise), each call passing the packed weights of the call after it as
its L2 prefetch range.  Weights are packed once before timing (offline step).

Metric: packed-weight GB/s (packed bytes streamed per step / step time).  The
same line carries, as nested objects: "decode_2b" (the same step on the 2B-class
shapes, M = 1 and 8, 30 layers), "prefill" (the M = 2048 prefill of the 8B
shapes 4096->14336 and 14336->4096 in int8-equivalent TOPS, 2 M N K / time) and
"stack_2b" (bitlinear_block_forward over the 30-layer linear stack of the
2B-class model at M = 1, 8 and 512).

    python bench.py [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload decode_8b|decode_2b|stack_2b]

The library drives one GPU: with --gpus N > 1 (under torchrun) rank 0 prints an
"unavailable" line and every rank exits 0.  The reference arm times the CPU
oracle (the plain single-threaded C definition) on a bounded sample of the same
workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import platform
import statistics
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "BitLinear decode packed-weight GB/s vs HBM peak; M=2048 prefill int8 TOPS"
HEADLINE = "decode_8b"
LAYERS = {"decode_8b": 32, "decode_2b": 30, "stack_2b": 30}
RMS_EPS = 1e-5


def log(*a):
    print(*a, file=sys.stderr, flush=True)


# ---------------------------------------------------------------------------
# environment helpers
# ---------------------------------------------------------------------------

def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")),
            int(os.environ.get("WORLD_SIZE", "1")))


def host_cpu():
    """CPU model of this host and the cores this process may run on."""
    model = platform.processor() or "unknown"
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.startswith("model name"):
                    model = line.split(":", 1)[1].strip()
                    break
    except OSError:
        pass
    try:
        avail = len(os.sched_getaffinity(0))
    except AttributeError:
        avail = os.cpu_count()
    return {"model": model, "nproc": avail}


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

_ORACLE_SAMPLE = {}


def _oracle_inputs(workload):
    """Layer 0 of a decode workload, ternarized by the oracle (offline step, not timed)."""
    if workload not in _ORACLE_SAMPLE:
        import oracle
        from bitlinear_rmsnorm_token_int8_b300 import synth
        wl = synth.WORKLOADS[workload]
        mats = []
        for pi, p in enumerate(wl.projections):
            W = synth.latent_weights(p.N, p.K, synth.weight_seed(wl.seed, 0, pi)).numpy()
            _, gamma, wq = oracle.pack_weights(W)
            del W
            mats.append((p, gamma, wq))
        xs = {}
        for M in wl.tokens:
            for K in sorted({p.K for p in wl.projections}):
                xs[(M, K)] = (synth.bf16_bits(synth.activations(M, K, synth.act_seed(wl.seed, M, K), outliers=False)),
                              synth.bf16_bits(synth.rms_gains(K, synth.gain_seed(wl.seed, 0, K))))
        _ORACLE_SAMPLE[workload] = (wl, mats, xs)
    return _ORACLE_SAMPLE[workload]


def oracle_sample(workload, seconds: float = 12.0):
    """Times the CPU oracle as it stands (act-quant + add/skip/subtract contraction +
    dequant) on layer 0 of the decode workload, every token count, projection by
    projection, until ~`seconds` have passed (at least one projection).  Returns
    (packed-weight GB/s, seconds, projections done, projections per pass)."""
    import oracle
    wl, mats, xs = _oracle_inputs(workload)
    calls = [(M, p, gamma, wq) for M in wl.tokens for (p, gamma, wq) in mats]
    done_bytes, n, t0 = 0, 0, time.perf_counter()
    while True:
        M, p, gamma, wq = calls[n % len(calls)]
        xb, gb = xs[(M, p.K)]
        xq, sig = oracle.act_quant(xb, gb, RMS_EPS)
        acc = oracle.ternary_matmul(xq, wq)
        oracle.dequant(acc, sig, np.full(p.N, float(gamma)))
        done_bytes += p.N * p.K // 4
        n += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    return done_bytes / el / 1e9, el, n, len(calls)


def reference_arm(args):
    rank, _, world = dist_env()
    if rank != 0:
        return 0
    import oracle
    oracle.build()
    workload = args.workload if args.workload != "stack_2b" else HEADLINE
    _oracle_inputs(workload)
    per_step = min(args.ref_seconds, 150.0 / max(args.steps, 1))   # whole arm within a few minutes
    t0 = time.perf_counter()
    gbs_list, done = [], 0
    for _ in range(args.steps):
        gbs, _, n, per_pass = oracle_sample(workload, per_step)
        gbs_list.append(gbs)
        done += n
    el = time.perf_counter() - t0
    value = float(statistics.mean(gbs_list))
    cpu = host_cpu()
    sample = (f"layer 0 of {LAYERS[workload]}: projections (QKV, O, gate+up, down) x tokens "
              f"{list(_ORACLE_SAMPLE[workload][0].tokens)} in turn, ~{per_step:.1f} s per step "
              f"({done} projection calls of {per_pass} per pass), single-threaded C oracle")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int32",
        "data": "synthetic", "config": {"workload": workload, "layers_sampled": 1},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": sample,
                         "host_cpu": cpu["model"], "host_nproc": cpu["nproc"]},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

def traffic_record(workload, kernel_srcs):
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
    r = rec.get(workload)
    if not r or r.get("source_sha") != sha:
        return None
    return float(r["dram_bytes_per_launch"])


def kernel_sources():
    csrc = os.path.join(ROOT, "bitlinear_rmsnorm_token_int8_b300", "csrc")
    return [os.path.join(csrc, f) for f in ("decode_cc.cu", "decode_dp4a.cu", "quant_math.cuh", "decode_tc.cu",
                                            "device_util.cuh", "act_ops.cuh")]


def timed_replays(torch, graph, stream, steps):
    """ms per replay of `graph`, by CUDA events on `stream` (the caller makes it current)."""
    assert torch.cuda.current_stream() == stream
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        graph.replay()
    e1.record(stream)
    stream.synchronize()
    return e0.elapsed_time(e1) / steps


def measure_decode(bl, synth, torch, dev, workload, layers, steps, warmup, e2e=True, clocks=True,
                   min_warmup_s=1.0):
    """The decode step of `workload` (see the module docstring) as one CUDA graph:
    value, step time, per-shape launch times and roofline, and the end-to-end pass."""
    wl = synth.WORKLOADS[workload]

    # ---- weights (offline step, not timed)
    weights = []
    for layer in range(layers):
        row = []
        for pi, p in enumerate(wl.projections):
            W = synth.latent_weights_device(p.N, p.K, synth.weight_seed(wl.seed, layer, pi), dev)
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

    # the calls of one step in order; each one's L2 prefetch is the next one's weights
    calls = [(M, li, pi) for M in wl.tokens for li in range(layers) for pi in range(len(wl.projections))]
    nxt = {calls[i]: calls[(i + 1) % len(calls)] for i in range(len(calls))}
    packed_bytes_step = sum(weights[li][pi][0].N * weights[li][pi][0].K // 4 for (_, li, pi) in calls)

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

    def layer(M, x, li, pi, y, prefetch):
        # one BitLinear layer through the public one-call API (RMSNorm + quantization +
        # contraction): one kernel for one token, quantization + contraction otherwise
        p, packed, w_scale = weights[li][pi]
        bl.bitlinear_linear_forward(x, gains[p.K], RMS_EPS, packed, w_scale, out_dtype=torch.bfloat16, y=y,
                                    workspace=lws[(M, p.N, p.K)], flags=FL, stream=stream, prefetch=prefetch)

    def step():
        """One pass: for each token count, layer and projection, the BitLinear layer."""
        for (M, li, pi) in calls:
            p = weights[li][pi][0]
            _, nli, npi = nxt[(M, li, pi)]
            layer(M, xs[(M, p.K)], li, pi, ys[(M, p.N)], weights[nli][npi][1])

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
    while n < warmup or time.perf_counter() - t0 < min_warmup_s:
        graph.replay()
        n += 1
        if n % 20 == 0:
            torch.cuda.synchronize()
    torch.cuda.synchronize()

    # ---- timed region: K replays of the step
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    clk = ClockSampler(dev.index or 0) if clocks else None
    if clk:
        clk.__enter__()
    with torch.cuda.stream(stream):
        start.record(stream)
        for _ in range(steps):
            graph.replay()
        end.record(stream)
    torch.cuda.synchronize()
    if clk:
        clk.__exit__(None, None, None)
    ms = start.elapsed_time(end) / steps
    value = packed_bytes_step / (ms * 1e-3) / 1e9
    assert bl.bitlinear_get_device_error() == 0

    # ---- per-launch durations of the kernel that does each projection's contraction
    #      (for one token with K <= 8192 the layer kernel, which also quantizes).  For
    #      each (M, projection) a CUDA graph holds the layers' launches back to back
    #      (distinct weights, each launch prefetching the next one's, chained by
    #      programmatic dependent launch as in the step); CUDA events on the launching
    #      stream bracket K replays, so the average is the kernel's duration in a stream
    #      of launches, not host launch latency.  Codes, scales and operand planes for
    #      the contraction-only launches come from one quantization per (M, K) beforehand.
    with torch.cuda.stream(stream):
        for M in wl.tokens:
            for K in Ks:
                bl.bitlinear_quant_act(xs[(M, K)], gains[K], RMS_EPS, x_q=xq[(M, K)], act_scale=sc[(M, K)],
                                       x_ops=ops[(M, K)], stream=stream)
    shape_graphs = []
    with torch.cuda.stream(stream):
        for M in wl.tokens:
            for pi, p in enumerate(wl.projections):
                def chain(M=M, pi=pi, p=p):
                    for li in range(layers):
                        nxt_packed = weights[(li + 1) % layers][pi][1]
                        if route(M, p) == bl.ROUTE_FUSED:    # the layer is one kernel
                            layer(M, xs[(M, p.K)], li, pi, ys[(M, p.N)], nxt_packed)
                        else:                                  # the contraction kernel alone
                            _, packed, w_scale = weights[li][pi]
                            codes = route(M, p) == bl.ROUTE_CODES
                            bl.bitlinear_forward(xq[(M, p.K)] if codes else None, sc[(M, p.K)], packed, w_scale,
                                                 out_dtype=torch.bfloat16, y=ys[(M, p.N)],
                                                 x_ops=None if codes else ops[(M, p.K)], K=p.K, flags=FL,
                                                 stream=stream, prefetch=nxt_packed)
                chain()
                stream.synchronize()
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream):
                    chain()
                shape_graphs.append((M, p, g))
        for _, _, g in shape_graphs:
            for _ in range(max(warmup, 3)):
                g.replay()
        stream.synchronize()
    hbm, _, peak_src = measured_peaks()
    per_shape, launch_ms, launch_bytes = [], [], []
    for M, p, g in shape_graphs:
        with torch.cuda.stream(stream):                  # replay on the stream the events record on
            per_launch = timed_replays(torch, g, stream, steps) / layers
        alg = alg_bytes(M, p)
        gbs = alg / (per_launch * 1e-3) / 1e9
        per_shape.append({"tokens": M, "projection": p.name, "K": p.K, "N": p.N,
                          "kernel": {bl.ROUTE_FUSED: "CUDA-core layer kernel (linear_dp4a / decode_cc)",
                                     bl.ROUTE_CODES: "CUDA-core codes kernel (decode_dp4a / decode_cc)"}.get(
                                         route(M, p), "decode_tc_kernel"),
                          "launch_us": per_launch * 1e3, "alg_bytes": alg, "alg_gbs": gbs, "frac": gbs / hbm})
        launch_ms.extend([per_launch] * layers)
        launch_bytes.extend([alg] * layers)
    achieved = sum(launch_bytes) / (sum(launch_ms) * 1e-3) / 1e9
    roofline = {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                "traffic": traffic_record(workload, kernel_sources()), "peak_source": peak_src,
                "kernel": "the decode contraction + dequant of each projection (per_shape[].kernel): for one "
                          "or two tokens decode_cc_kernel (CUDA cores; for K <= 8192 the whole layer: RMSNorm, "
                          "quantization, int8-code contraction), for more decode_tc_kernel (tcgen05)",
                "timing": "CUDA events around K replays of a graph of the layers' launches per (M, projection)",
                "alg_bytes_per_launch": sum(launch_bytes) / len(launch_bytes),
                "avg_launch_us": sum(launch_ms) / len(launch_ms) * 1e3,
                "share_of_step": sum(launch_ms) / ms if ms > 0 else None,
                "per_shape": per_shape}
    out = {"workload": workload, "layers": layers, "tokens": list(wl.tokens),
           "projections": [[p.name, p.K, p.N] for p in wl.projections], "value": value, "unit": "GB/s",
           "ms_per_step": ms, "packed_bytes_per_step": packed_bytes_step,
           "gpu_launches": int(launches_per_step * steps), "launches_per_step": int(launches_per_step),
           "roofline": roofline, "clocks": clk.summary() if clk else None}
    if not e2e:
        del shape_graphs, graph
        return out

    # ---- end to end through the public API: pinned host inputs in, bf16 outputs out.
    #      Every projection of the step gets its own input rows; they travel to the
    #      device as one copy per token count from one pinned buffer, and each layer's
    #      outputs come back as one copy, the way a caller stages a step's data.
    in_off, out_off = {}, {}
    h2d = d2h = 0
    for (M, li, pi) in calls:
        p = weights[li][pi][0]
        in_off[(M, li, pi)] = h2d // 2
        out_off[(M, li, pi)] = d2h // 2
        h2d += M * p.K * 2
        d2h += M * p.N * 2
    host_in = torch.empty(h2d // 2, dtype=torch.bfloat16, pin_memory=True)
    host_out = torch.empty(d2h // 2, dtype=torch.bfloat16, pin_memory=True)
    for (M, li, pi) in calls:
        p = weights[li][pi][0]
        o = in_off[(M, li, pi)]
        host_in[o:o + M * p.K].copy_(xs[(M, p.K)].reshape(-1).cpu())
    dev_in = torch.empty_like(host_in, device=dev)
    dev_out = torch.empty_like(host_out, device=dev)
    last_p = len(wl.projections) - 1
    in_rng = {M: (in_off[(M, 0, 0)], in_off[(M, layers - 1, last_p)] + M * wl.projections[-1].K) for M in wl.tokens}
    out_rng = {(M, li): (out_off[(M, li, 0)], out_off[(M, li, last_p)] + M * wl.projections[-1].N)
               for M in wl.tokens for li in range(layers)}
    side = torch.cuda.Stream(device=dev)       # host<->device copies, beside the kernels

    def e2e_step():
        """Inputs in, per projection RMSNorm + quant and the contraction, outputs out.  The
        copies run on a side stream: each token count's inputs as one copy (the later ones
        while the earlier pass computes), each layer's outputs as soon as it is done."""
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
            for li in range(layers):
                for pi, p in enumerate(wl.projections):
                    o = in_off[(M, li, pi)]
                    yo = out_off[(M, li, pi)]
                    _, nli, npi = nxt[(M, li, pi)]
                    layer(M, dev_in[o:o + M * p.K].view(M, p.K), li, pi, dev_out[yo:yo + M * p.N].view(M, p.N),
                          weights[nli][npi][1])
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
        for _ in range(max(warmup, 1)):
            e2e_graph.replay()
        torch.cuda.synchronize()
        e2e_ms = timed_replays(torch, e2e_graph, stream, steps)
    out["e2e"] = {"value": packed_bytes_step / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s", "h2d_bytes_per_step": h2d,
                  "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms}
    del shape_graphs, graph, e2e_graph
    return out


def measure_prefill(bl, synth, torch, dev, steps, warmup, peaks=None):
    """M = 2048 prefill of the 8B-class shapes (4096->14336, 14336->4096): per shape one
    graph of the whole BitLinear layer (bitlinear_linear_forward: RMSNorm + quantization
    into the operand form, then the contraction); CUDA events around `steps` replays.
    Reports int8-equivalent TOPS (2 M N K / time) of the quant + contraction pair and of
    the contraction alone.  The contraction issues two e4m3 MMAs per int8 product (each
    code is two exact e4m3 planes), so its tensor pipe runs 4 M N K e4m3 FLOP: the
    roofline fraction counts the method's 2 M N K against the e4m3 peak, and
    mma_pipe_frac the MMA work actually issued."""
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
        cl = bl.bitlinear_prefill_cluster_size(ops, M, p.N, p.K)
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
                ms[kind] = timed_replays(torch, gr, stream, steps)
        ops_ = 2.0 * M * p.N * p.K
        out["shapes"].append({"K": p.K, "N": p.N, "ms": ms["pair"], "fwd_ms": ms["fwd"], "cluster": cl,
                              "int8_equiv_tops": ops_ / (ms["pair"] * 1e9),
                              "fwd_int8_equiv_tops": ops_ / (ms["fwd"] * 1e9)})
        tot_ops += ops_
        tot_ms += ms["pair"]
        tot_fwd_ms += ms["fwd"]
        del packed, w_scale, x, ops, ws, y, graphs
    method_tops = tot_ops / (tot_fwd_ms * 1e9)
    layer_tops = tot_ops / (tot_ms * 1e9)
    pk = peaks or {}
    if "tcgen05_e4m3_tflops" in pk:
        fp8_peak, src = pk["tcgen05_e4m3_tflops"], "measured (tcgen05 kind::f8f6f4 m128n256k32 microbenchmark)"
    else:
        _, bf16_tf, s = measured_peaks()
        fp8_peak, src = 2.0 * bf16_tf, f"{s} bf16 cuBLAS x 2 (nominal e4m3:bf16 ratio)"
    out.update({"int8_equiv_tops": layer_tops, "fwd_int8_equiv_tops": method_tops,
                "roofline": {"bound": "tensor", "achieved": method_tops,
                             "unit": "TFLOP/s (int8-equivalent method work, 2 M N K)",
                             "peak": fp8_peak, "frac": method_tops / fp8_peak,
                             "mma_pipe_frac": 2.0 * method_tops / fp8_peak,
                             "layer_frac": layer_tops / fp8_peak,
                             "kernel": "prefill_tc_kernel (tcgen05 kind::f8f6f4, two e4m3 MMAs per int8 product)",
                             "peak_source": src}})
    if "mma_sync_s8_tops" in pk:
        out["vs_int8_mma_sync"] = {"peak_tops": pk["mma_sync_s8_tops"],
                                   "ratio": method_tops / pk["mma_sync_s8_tops"],
                                   "note": "the only int8 tensor-core MMA on this GPU (tcgen05 kind::i8 is "
                                           "rejected for sm_103a)"}
    return out


def measure_mma_peaks(torch, dev):
    """Dense MMA rates from libbitlinear_probe.so (back-to-back MMAs on on-chip
    operands, one CTA per SM for tcgen05), by CUDA events, with the SM clock seen."""
    import ctypes
    path = os.path.join(ROOT, "bitlinear_rmsnorm_token_int8_b300", "libbitlinear_probe.so")
    if not os.path.exists(path):
        return None
    L = ctypes.CDLL(path)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    ms = ctypes.c_float()
    out = {}
    with ClockSampler(dev.index or 0) as clk:
        for kind, key, flop in ((0, "tcgen05_e4m3_tflops", 2 * 128 * 256 * 32),
                                (1, "tcgen05_bf16_tflops", 2 * 128 * 256 * 16)):
            iters = 16384
            if L.bitlinear_probe_tcgen05(kind, iters, sms, ctypes.byref(ms)) == 0:
                out[key] = flop * iters * sms / (ms.value * 1e-3) / 1e12
        for kind, key in ((0, "mma_sync_s8_tops"), (1, "mma_sync_e4m3_tflops")):
            iters, ctas = 2048, sms * 8
            if L.bitlinear_probe_mma_sync(kind, iters, ctas, ctypes.byref(ms)) == 0:
                out[key] = 2 * 16 * 8 * 32 * 8 * iters * ctas * 8 / (ms.value * 1e-3) / 1e12
    out["clocks"] = clk.summary()
    out["how"] = ("tcgen05: m128n256 MMAs, A in tensor memory, B in shared memory, 16384 per CTA on one CTA per "
                  "SM; mma.sync: m16n8k32, 8 warps x 8 independent accumulators, 8 CTAs per SM")
    return out


def measure_stack(bl, synth, torch, dev, layers, steps, warmup):
    """30-layer BitLinear stack (bitlinear_block_forward) at M = 1, 8 and 512 tokens."""
    wl = synth.WORKLOADS["stack_2b"]
    H, NQKV, F = 2560, 3840, 6912
    layer_list, packed_bytes = [], 0
    for l in range(layers):
        layer = {}
        for j, (name, shapes) in enumerate({"qkv": [(NQKV, H)], "o": [(H, H)], "gate_up": [(F, H), (F, H)],
                                            "down": [(H, F)]}.items()):
            Ws = [synth.latent_weights_device(n, k, synth.weight_seed(wl.seed, l, 3 * j + i), dev)
                  for i, (n, k) in enumerate(shapes)]
            layer[name], layer[name + "_scale"] = bl.pack_stacked(Ws)
            packed_bytes += sum(n * k // 4 for n, k in shapes)
            del Ws
        for j, (name, k) in enumerate({"gain_qkv": H, "gain_o": H, "gain_gate_up": H, "gain_down": F}.items()):
            layer[name] = synth.rms_gains(k, synth.gain_seed(wl.seed, l, j)).to(dev)
        layer_list.append(layer)
    torch.cuda.synchronize()
    stream = torch.cuda.Stream(device=dev)
    results = {}
    for M in wl.tokens:
        x0 = synth.activations(M, H, synth.act_seed(wl.seed, M, H), outliers=True).to(dev)
        x = x0.clone()
        ws = torch.empty(bl.bitlinear_block_workspace_bytes(M, H, NQKV, F) + 256, dtype=torch.uint8, device=dev)
        with torch.cuda.stream(stream):
            bl.bitlinear_block_forward(layer_list, x, H, NQKV, F, RMS_EPS, workspace=ws, flags=bl.FLAG_PDL,
                                       stream=stream)
            stream.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                bl.bitlinear_block_forward(layer_list, x, H, NQKV, F, RMS_EPS, workspace=ws, flags=bl.FLAG_PDL,
                                           stream=stream)
            for _ in range(max(warmup, 3)):
                g.replay()
            ms = timed_replays(torch, g, stream, steps)
        assert bl.bitlinear_get_device_error(stream) == 0
        results[str(M)] = {"ms_per_forward": ms, "tokens_per_s": M / (ms * 1e-3),
                           "packed_gbs": packed_bytes / (ms * 1e-3) / 1e9,
                           "int8_equiv_tops": 2.0 * M * 4 * packed_bytes / (ms * 1e9)}
    return {"workload": "stack_2b", "layers": layers, "hidden": H, "qkv": NQKV, "ffn": F,
            "packed_bytes_per_forward": packed_bytes, "per_tokens": results}


def our_arm(args):
    import torch
    import bitlinear_rmsnorm_token_int8_b300 as bl
    from bitlinear_rmsnorm_token_int8_b300 import synth

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    bl.lib()
    workload = args.workload
    if workload == "stack_2b":
        st = measure_stack(bl, synth, torch, dev, args.layers or LAYERS["stack_2b"], args.steps, args.warmup)
        m1 = st["per_tokens"]["1"]
        print(json.dumps({"metric": METRIC, "value": m1["packed_gbs"], "unit": "GB/s", "n_gpus": 1,
                          "steps": args.steps, "warmup": args.warmup, "ms_per_step": m1["ms_per_forward"],
                          "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int32",
                          "data": "synthetic", "config": {"workload": "stack_2b"}, "stack_2b": st}), flush=True)
        return 0

    head = measure_decode(bl, synth, torch, dev, workload, args.layers or LAYERS[workload], args.steps,
                          args.warmup, e2e=True, clocks=True, min_warmup_s=args.min_warmup_s)
    extra = {}
    if workload == HEADLINE and not args.headline_only:
        d2 = measure_decode(bl, synth, torch, dev, "decode_2b", LAYERS["decode_2b"], args.steps, args.warmup,
                            e2e=False, clocks=False)
        extra["decode_2b"] = {k: d2[k] for k in ("value", "unit", "ms_per_step", "layers", "tokens",
                                                 "packed_bytes_per_step")}
        extra["decode_2b"]["roofline"] = {k: d2["roofline"][k] for k in ("achieved", "frac", "avg_launch_us",
                                                                         "per_shape")}
        torch.cuda.empty_cache()
        extra["mma_peaks"] = measure_mma_peaks(torch, dev)
        extra["prefill"] = measure_prefill(bl, synth, torch, dev, max(3, args.steps), args.warmup,
                                           peaks=extra["mma_peaks"])
        torch.cuda.empty_cache()
        extra["stack_2b"] = measure_stack(bl, synth, torch, dev, LAYERS["stack_2b"], max(3, args.steps // 2),
                                          args.warmup)

    cpu = None
    if not args.no_cpu_baseline:
        gbs, el, n, per_pass = oracle_sample(workload, args.ref_seconds)
        hc = host_cpu()
        cpu = {"value": gbs, "unit": "GB/s", "cores": 1, "kind": "oracle",
               "sample": f"layer 0 of {head['layers']}: (tokens, projection) calls of one pass in turn, "
                         f"{n} of {per_pass} per pass in {el:.1f} s, single-threaded C oracle",
               "host_cpu": hc["model"], "host_nproc": hc["nproc"]}

    wl = synth.WORKLOADS[workload]
    line = {
        "metric": METRIC, "value": head["value"], "unit": "GB/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": head["ms_per_step"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "int32",
        "data": "synthetic (seeded N(0,0.02) latent weights, N(0,1) bf16 activations)",
        "config": {"workload": workload, "layers": head["layers"], "tokens": list(wl.tokens),
                   "projections": head["projections"], "packed_bytes_per_step": head["packed_bytes_per_step"],
                   "l2": f"no flush: {head['packed_bytes_per_step'] / len(wl.tokens) / 1e6:.0f} MB of distinct "
                         "packed weights per token-count pass (> 4x the 126 MB L2)",
                   "launch": "one CUDA graph per step; kernels chained by programmatic dependent launch; "
                             "each call prefetches the next call's weights into L2",
                   "parallelism": "single GPU"},
        "e2e": {k: head["e2e"][k] for k in ("value", "unit", "h2d_bytes_per_step", "d2h_bytes_per_step")},
        "gpu_launches": head["gpu_launches"],
        "roofline": head["roofline"],
        "cpu_baseline": cpu,
        "clocks": head["clocks"],
    }
    line.update(extra)
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--layers", type=int, default=0, help="layers of the workload (default: its own)")
    ap.add_argument("--ref-seconds", type=float, default=12.0, help="CPU oracle seconds per sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--min-warmup-s", type=float, default=2.0,
                    help="warm-up replays continue at least this long (clock ramp-up; 0 under a profiler)")
    ap.add_argument("--headline-only", action="store_true",
                    help="only the headline decode (no decode_2b, prefill or stack_2b objects)")
    ap.add_argument("--workload", choices=["decode_8b", "decode_2b", "stack_2b"], default=HEADLINE)
    args = ap.parse_args()
    rank, _, world = dist_env()
    if args.impl == "reference":
        return reference_arm(args)
    if world > 1 or args.gpus > 1:
        if rank == 0:
            print(json.dumps({"metric": METRIC, "n_gpus": max(world, args.gpus),
                              "unavailable": "one-GPU library: the BitLinear forward runs on a single GPU "
                                             "(no multi-GPU path)"}), flush=True)
        return 0
    return our_arm(args)


if __name__ == "__main__":
    sys.exit(main())
