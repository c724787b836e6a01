"""Single-shape runs of the hot path, for profilers (ncu) and quick timing.

    python -m bitlinear_rmsnorm_token_int8_b300.cases forward M K N [reps] [route]
        one BitLinear projection: quantize M x K activations once, then `reps`
        contractions against one packed N x K weight.  route: `auto` (default: the
        library's choice given both x_q and the operand form: the int8-code kernel
        for one token (two with K <= 4096), the tcgen05 decode kernel up to 32
        tokens, the tcgen05 prefill kernel above), `ops` (operand form only:
        always a tcgen05 kernel), `codes` (x_q only) or `layer` (the one-call
        layer bitlinear_linear_forward on the bf16 activations: for one token
        with K <= 8192, or up to 16384 for large matrices, a single kernel that also quantizes).
    python -m bitlinear_rmsnorm_token_int8_b300.cases shapes WORKLOAD [reps]
        every (tokens, projection) shape of a named workload (synth.WORKLOADS),
        `reps` launches each of the kernel bench.py times for it (route `layer`
        where the layer is one kernel, else `auto`), every one on freshly packed
        weights (cold L2).

Inputs are seeded synthetic draws (synth); every call goes through the public
binding, and the run ends by checking the device error word.
"""
from __future__ import annotations

import sys

import torch

from . import (ROUTE_FUSED, bitlinear_forward, bitlinear_get_device_error, bitlinear_linear_forward,
               bitlinear_linear_route, bitlinear_pack_weights, bitlinear_quant_act)
from . import synth


def _one(M: int, K: int, N: int, reps: int, dev, fresh_weights: bool, route: str = "auto") -> None:
    x = synth.activations(M, K, seed=synth.act_seed(7, M, K)).to(dev)
    xq, sc, ops = bitlinear_quant_act(x, None, 1e-5, x_ops=True)
    if route == "ops":
        xq = None
    elif route == "codes":
        ops = None
    y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    packed = ws = None
    for r in range(reps):
        if packed is None or fresh_weights:
            W = synth.latent_weights_device(N, K, seed=synth.weight_seed(7, r, 0), device=dev)
            packed, ws, _ = bitlinear_pack_weights(W)
            del W
        if route == "layer":
            bitlinear_linear_forward(x, None, 1e-5, packed, ws, y=y)
        else:
            bitlinear_forward(xq, sc, packed, ws, y=y, x_ops=ops, K=K)
    torch.cuda.synchronize()


def main(argv: list[str]) -> int:
    if len(argv) < 2 or argv[0] not in ("forward", "shapes"):
        print(__doc__)
        return 2
    dev = torch.device("cuda", 0)
    if argv[0] == "forward":
        M, K, N = (int(a) for a in argv[1:4])
        reps = int(argv[4]) if len(argv) > 4 else 3
        route = argv[5] if len(argv) > 5 else "auto"
        if route not in ("auto", "ops", "codes", "layer"):
            print(__doc__)
            return 2
        _one(M, K, N, reps, dev, fresh_weights=False, route=route)
        print(f"forward M={M} K={K} N={N} x{reps} route={route}")
    else:
        wl = synth.WORKLOADS[argv[1]]
        reps = int(argv[2]) if len(argv) > 2 else 2
        for M in wl.tokens:
            for p in wl.projections:
                route = "layer" if bitlinear_linear_route(M, p.N, p.K) == ROUTE_FUSED else "auto"
                _one(M, p.K, p.N, reps, dev, fresh_weights=True, route=route)
                print(f"shape M={M} {p.name} K={p.K} N={p.N} x{reps}")
    err = bitlinear_get_device_error()
    if err != 0:
        print(f"device error word {err}")
        return 1
    return 0


if __name__ == "__main__":
    sys.exit(main(sys.argv[1:]))
