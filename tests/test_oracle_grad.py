"""Pins of the gradient oracle (CPU): its forward equals the numpy oracle's layer, its
gradients match central finite differences along random directions (no autodiff), and the
closed-form reverse chunk scan -- the structure the GPU backward follows -- reproduces them."""
import numpy as np
import pytest
import torch

from oracle import oracle
from oracle.oracle_grad import forward_torch, layer_backward
from weight_mlp_layers_swiglu_b300.inputs import random_case

NAMES = ["H", "X0", "W_gate", "W_up", "W_down0", "W_target", "conv_w"]


def _case(B=2, T=20, d=4, f=6, C=8, k=3, eta=0.7, seed=3):
    w, x = random_case(B, T, d, f, C, k, eta, "f32", seed)
    x = {n: t.double() for n, t in x.items()}
    g = torch.Generator().manual_seed(seed + 50)
    dO = torch.randn(B, T, d, generator=g, dtype=torch.float64)
    dWf = torch.randn(B, d, f, generator=g, dtype=torch.float64)
    return w, x, dO, dWf


def test_forward_matches_the_oracle():
    w, x, _, _ = _case()
    O, Wf = forward_torch(*(x[n] for n in NAMES), w.C, w.eta)
    O_ref, W_ref = oracle.layer_forward(*(x[n] for n in NAMES), w.C, w.eta)
    assert np.abs(O.numpy() - O_ref).max() < 1e-12 and np.abs(Wf.numpy() - W_ref).max() < 1e-12


@pytest.mark.parametrize("name", NAMES)
def test_gradient_matches_central_differences(name):
    w, x, dO, dWf = _case()
    grads = layer_backward(*(x[n] for n in NAMES), w.C, w.eta, dO, dWf)
    g = torch.Generator().manual_seed(99)
    v = torch.randn(x[name].shape, generator=g, dtype=torch.float64)

    def loss(xx):
        O, Wf = oracle.layer_forward(*(xx[n] for n in NAMES), w.C, w.eta)
        return float((O * dO.numpy()).sum() + (Wf * dWf.numpy()).sum())

    h = 1e-5
    xp, xm = dict(x), dict(x)
    xp[name] = x[name] + h * v
    xm[name] = x[name] - h * v
    fd = (loss(xp) - loss(xm)) / (2 * h)
    an = float((grads[name] * v).sum())
    assert abs(fd - an) <= 1e-6 * max(1.0, abs(an))


def test_reverse_chunk_scan_reproduces_autograd():
    """G_i = dO_i^T Z_i; R_i = dW_final + sum_{l>i} G_l (exclusive suffix); dZ_i = dO_i W_i + eta V_i R_i;
    dV_i = eta Z_i R_i^T; dW_down0 = sum over sequences of (dW_final + sum_i G_i)."""
    w, x, dO, dWf = _case(B=2, T=29, C=8)
    grads = layer_backward(*(x[n] for n in NAMES), w.C, w.eta, dO, dWf)
    W0 = x["W_down0"].numpy()
    dW0 = np.zeros_like(W0)
    for b in range(w.B):
        Z = oracle.swiglu(x["H"][b], x["W_gate"], x["W_up"])
        V = oracle.target(x["X0"][b], x["conv_w"], x["W_target"])
        W_eff, _ = oracle.chunk_weights(V, Z, W0, w.C, w.eta)
        rows = oracle.chunk_rows(w.T, w.C)
        G = [dO[b, lo:hi].numpy().T @ Z[lo:hi] for lo, hi in rows]
        R = [dWf[b].numpy() + sum(G[i + 1:], np.zeros_like(W0)) for i in range(len(rows))]
        dZ = np.zeros_like(Z)
        dV = np.zeros_like(V)
        for i, (lo, hi) in enumerate(rows):
            dZ[lo:hi] = dO[b, lo:hi].numpy() @ W_eff[i] + w.eta * V[lo:hi] @ R[i]
            dV[lo:hi] = w.eta * Z[lo:hi] @ R[i].T
        dW0 += dWf[b].numpy() + sum(G, np.zeros_like(W0))
        # through the target projection: dY = dV W_target^T, and the causal conv's adjoint
        dY = dV @ x["W_target"].numpy().T
        k = w.k
        dX0 = np.zeros((w.T, w.d))
        for s in range(k):
            back = k - 1 - s
            dX0[: w.T - back] += x["conv_w"].numpy()[:, s] * dY[back:]
        assert np.abs(dX0 - grads["X0"][b].numpy()).max() < 1e-10
        # through the gated MLP
        A = x["H"][b].numpy() @ x["W_gate"].numpy().T
        U = x["H"][b].numpy() @ x["W_up"].numpy().T
        sg = 1 / (1 + np.exp(-A))
        dA = dZ * U * sg * (1 + A * (1 - sg))
        dU = dZ * A * sg
        dH = dA @ x["W_gate"].numpy() + dU @ x["W_up"].numpy()
        assert np.abs(dH - grads["H"][b].numpy()).max() < 1e-10
    assert np.abs(dW0 - grads["W_down0"].numpy()).max() < 1e-10
