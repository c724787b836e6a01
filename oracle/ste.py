"""Straight-through estimator (STE) of the ternary weight quantizer, for the
training-side gradient check.

TEST INFRASTRUCTURE ONLY, like the rest of ``oracle/``: the CUDA library computes
the forward pass and has no backward.  Each function names the passage it follows:

* [P5-ste] "BitNet 1-bit LLM Inference Framework", section "Straight-Through
  Estimator (STE)": the forward pass ternarizes the weights, the backward pass
  hands the incoming gradient to the full-precision weights unchanged.
* [P1-ste] "BitNet's 1-Bit Transformer: Architecture Breakdown", section "Core
  Modifications", item 2: dL/dW = dL/dW_bit x clip(dW_bit/dW, -1, 1).  READING:
  the straight-through surrogate of dW_bit/dW is 1, and clip(1, -1, 1) = 1, so
  the clipped form passes the gradient unchanged as well.
* [P4-code] "BitNet b1.58 in Production: 1-Bit LLMs and Energy Benchmarks",
  bit_linear.py BitLinear.forward: the same estimator written as
  w + (w_q - w).detach() (and likewise for the activations).
"""
from __future__ import annotations

import numpy as np
import torch

from . import EPS_W, absmean_gamma, ternarize


class TernarySTE(torch.autograd.Function):
    """[P5-ste] forward: W_q = Clip(Round(W / (gamma + eps)), -1, 1) (the oracle's
    ternarize, float64 out); backward: the gradient passes straight through."""

    @staticmethod
    def forward(ctx, w: torch.Tensor, gamma: float, eps: float):
        q = ternarize(w.detach().cpu().numpy().astype(np.float32), np.float32(gamma), np.float32(eps))
        return torch.from_numpy(q.astype(np.float64))

    @staticmethod
    def backward(ctx, grad_out: torch.Tensor):
        return grad_out, None, None


def ternary_ste(w: torch.Tensor, eps: float = float(EPS_W)) -> torch.Tensor:
    """Ternary codes of w (float64) with the absmean gamma of w, through :class:`TernarySTE`."""
    gamma = absmean_gamma(w.detach().cpu().numpy().astype(np.float32))
    return TernarySTE.apply(w, float(gamma), eps)


def clipped_ste_grad(grad_wbit: torch.Tensor, surrogate: torch.Tensor | float = 1.0) -> torch.Tensor:
    """[P1-ste] dL/dW = dL/dW_bit * clip(dW_bit/dW, -1, 1), with the straight-through
    surrogate dW_bit/dW = 1 unless another one is given."""
    return grad_wbit * torch.clamp(torch.as_tensor(surrogate, dtype=grad_wbit.dtype), -1.0, 1.0)


def detach_ste(w: torch.Tensor, w_q: torch.Tensor) -> torch.Tensor:
    """[P4-code] w + (w_q - w).detach(): the value of w_q, the gradient of w."""
    return w + (w_q - w).detach()
