"""Seeded synthetic inputs shaped like BitNet b1.58 BitLinear workloads.

This module holds only random-number generation and shape tables: none of the
method's arithmetic.  Both the CUDA path (through the tests and ``bench.py``)
and the CPU oracle are fed from here, so the two always see the same bytes.

Distributions (BitNet-shaped, no trained checkpoints exist offline):

* latent weights: fp32 N(0, 0.02^2)
* activations:    fp32 N(0, 1), optionally 1% of entries multiplied by 20
                  (outliers), rounded to bf16 (nearest even)
* RMSNorm gains:  bf16 U(0.5, 1.5)

All draws use a CPU ``torch.Generator`` seeded per tensor, so they do not depend
on the device or on what was drawn before.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

WEIGHT_STD = 0.02
OUTLIER_FRACTION = 0.01
OUTLIER_SCALE = 20.0


def _gen(seed: int) -> torch.Generator:
    return torch.Generator(device="cpu").manual_seed(int(seed))


def latent_weights(N: int, K: int, seed: int, std: float = WEIGHT_STD) -> torch.Tensor:
    """fp32 [N, K] (out x in, nn.Linear layout) ~ N(0, std^2)."""
    return torch.randn(N, K, generator=_gen(seed), dtype=torch.float32) * std


def activations(M: int, K: int, seed: int, outliers: bool = True) -> torch.Tensor:
    """bf16 [M, K] ~ N(0,1); with ``outliers`` 1% of entries are scaled by 20."""
    g = _gen(seed)
    x = torch.randn(M, K, generator=g, dtype=torch.float32)
    if outliers:
        mask = torch.rand(M, K, generator=g) < OUTLIER_FRACTION
        x = torch.where(mask, x * OUTLIER_SCALE, x)
    return x.to(torch.bfloat16)


def rms_gains(K: int, seed: int, lo: float = 0.5, hi: float = 1.5) -> torch.Tensor:
    """bf16 [K] ~ U(lo, hi)."""
    return (torch.rand(K, generator=_gen(seed), dtype=torch.float32) * (hi - lo) + lo).to(torch.bfloat16)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """Raw uint16 bit patterns of a CPU bf16 tensor (for the oracle)."""
    assert t.dtype == torch.bfloat16
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


# ---------------------------------------------------------------------------
# workload shapes
# ---------------------------------------------------------------------------

@dataclass(frozen=True)
class Projection:
    name: str
    K: int   # in features
    N: int   # out features


@dataclass(frozen=True)
class Workload:
    name: str
    tokens: tuple
    projections: tuple
    outliers: bool
    out_dtype: str
    seed: int
    layers: int = 1
    note: str = ""
    extra: dict = field(default_factory=dict)


# hidden 2560, FFN 6912 (2B class); hidden 4096, FFN 14336 (8B class)
PROJ_2B = (Projection("qkv", 2560, 3840), Projection("o", 2560, 2560),
           Projection("gate_up", 2560, 2 * 6912), Projection("down", 6912, 2560))
PROJ_8B = (Projection("qkv", 4096, 6144), Projection("o", 4096, 4096),
           Projection("gate_up", 4096, 2 * 14336), Projection("down", 14336, 4096))

WORKLOADS = {
    "single_k256_n512_m4": Workload(
        "single_k256_n512_m4", (4,), (Projection("single", 256, 512),), True, "f32", 1000),
    "decode_2b": Workload(
        "decode_2b", (1, 8), PROJ_2B, False, "bf16", 1001),
    "decode_8b": Workload(
        "decode_8b", (1, 4, 16), PROJ_8B, False, "bf16", 1002),
    "prefill_8b_m2048": Workload(
        "prefill_8b_m2048", (2048,), (Projection("up_4096_14336", 4096, 14336),
                                      Projection("down_14336_4096", 14336, 4096)), True, "bf16", 1003),
    "stack_2b": Workload(
        "stack_2b", (1, 8, 512), PROJ_2B, True, "bf16", 1004, layers=30,
        note="30 layers, hidden 2560, FFN 6912, ReLU^2 gating"),
}


def weight_seed(workload_seed: int, layer: int, proj_index: int) -> int:
    return workload_seed * 100003 + layer * 101 + proj_index


def act_seed(workload_seed: int, M: int, K: int) -> int:
    return workload_seed * 7919 + M * 31 + K


def gain_seed(workload_seed: int, layer: int, which: int) -> int:
    return workload_seed * 50021 + layer * 11 + which


def latent_weights_device(N: int, K: int, seed: int, device, std: float = WEIGHT_STD) -> torch.Tensor:
    """Same distribution as :func:`latent_weights`, drawn on ``device`` (for large benchmark
    stacks; the values differ from the CPU draw, the distribution does not)."""
    g = torch.Generator(device=device).manual_seed(int(seed))
    return torch.randn(N, K, generator=g, dtype=torch.float32, device=device) * std
