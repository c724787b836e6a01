"""The straight-through estimator of the ternary weight quantizer (CPU only; the
CUDA library has no backward).  Pins: the forward equals the oracle's
ternarization; the backward is the identity on the incoming gradient, exactly;
the clipped form of "BitNet's 1-Bit Transformer" reduces to it; and a linear
layer's weight gradient through the STE equals the closed form G^T X of the
same layer with the quantized weights held as values."""
import numpy as np
import torch

import oracle
from oracle import ste


def test_forward_is_the_ternarization():
    rng = np.random.default_rng(0)
    w = torch.from_numpy((rng.standard_normal((7, 12)) * 0.02).astype(np.float32)).double()
    q = ste.ternary_ste(w)
    _, _, o_q = oracle.pack_weights(w.float().numpy())
    assert (q.numpy() == o_q).all()
    assert set(np.unique(q.numpy())) <= {-1.0, 0.0, 1.0}


def test_backward_passes_the_gradient_unchanged():
    rng = np.random.default_rng(1)
    w = torch.from_numpy((rng.standard_normal((5, 8)) * 0.02).astype(np.float32)).double().requires_grad_(True)
    g = torch.from_numpy(rng.standard_normal((5, 8)))
    q = ste.ternary_ste(w)
    q.backward(g)
    assert torch.equal(w.grad, g)                    # exactly the incoming gradient, even where W_q = 0


def test_clipped_form_reduces_to_identity():
    g = torch.tensor([-3.0, -0.5, 0.0, 0.25, 7.0], dtype=torch.float64)
    assert torch.equal(ste.clipped_ste_grad(g), g)
    # a surrogate outside [-1, 1] is clipped: the gradient is never amplified
    assert torch.equal(ste.clipped_ste_grad(g, 4.0), g)
    assert torch.equal(ste.clipped_ste_grad(g, -2.5), -g)


def test_linear_weight_gradient_through_the_ste_matches_closed_form():
    # y = (X W_q^T) s with W_q from the STE: dL/dW = s G^T X, the gradient of the
    # full-precision weights as if W_q were W (the detach form gives the same)
    rng = np.random.default_rng(2)
    M, N, K = 3, 6, 10
    X = torch.from_numpy(rng.integers(-127, 128, (M, K)).astype(np.float64))
    s = 0.0123
    G = torch.from_numpy(rng.standard_normal((M, N)))
    w = torch.from_numpy((rng.standard_normal((N, K)) * 0.02).astype(np.float32)).double()
    for form in ("function", "detach"):
        wv = w.clone().requires_grad_(True)
        q = ste.ternary_ste(wv) if form == "function" else ste.detach_ste(wv, ste.ternary_ste(wv).detach())
        y = (X @ q.T) * s
        y.backward(G)
        assert torch.allclose(wv.grad, s * G.T @ X, rtol=0, atol=1e-12)
        assert torch.equal(y.detach(), (X @ ste.ternary_ste(w).T) * s)
