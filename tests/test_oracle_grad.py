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


@pytest.mark.parametrize("variant", ["no_proj", "shift"])
@pytest.mark.parametrize("name", ["H", "X0", "W_down0", "conv_w"])
def test_variant_gradients_match_central_differences(variant, name):
    """The ablation variants (identity projection; conv window ending at the next token) against
    finite differences of the numpy oracle's own variant forward."""
    w, x, dO, dWf = _case(T=19)
    shift = 1 if variant == "shift" else 0
    if variant == "no_proj":
        x["W_target"] = None
    grads = layer_backward(*(x[n] for n in NAMES), w.C, w.eta, dO, dWf, shift=shift)
    assert (grads["W_target"] is None) == (variant == "no_proj")
    v = torch.randn(x[name].shape, generator=torch.Generator().manual_seed(7), dtype=torch.float64)

    def loss(xx):
        O, Wf = oracle.layer_forward(*(xx[n] for n in NAMES), w.C, w.eta, shift=shift)
        return float((O * dO.numpy()).sum() + (Wf * dWf.numpy()).sum())

    h = 1e-5
    xp, xm = dict(x), dict(x)
    xp[name] = x[name] + h * v
    xm[name] = x[name] - h * v
    fd = (loss(xp) - loss(xm)) / (2 * h)
    an = float((grads[name] * v).sum())
    assert abs(fd - an) <= 1e-6 * max(1.0, abs(an))


def test_shifted_conv_adjoint_by_brute_force():
    """dX0 of the shifted variant is the transpose of the shifted conv, built as an explicit
    [T, T] matrix per channel, applied to the gradient that reaches V (identity projection)."""
    w, x, dO, _ = _case(B=1, T=11, d=3, f=4, C=4, k=3)
    x["W_target"] = None
    grads = layer_backward(*(x[n] for n in NAMES), w.C, w.eta, dO, None, shift=1)
    k, T = w.k, w.T
    cw = x["conv_w"]
    # the gradient w.r.t. V, from the chunk loop written with V as the free variable
    V = torch.zeros(T, w.d, dtype=torch.float64, requires_grad=True)
    A = x["H"][0] @ x["W_gate"].T
    Z = A * torch.sigmoid(A) * (x["H"][0] @ x["W_up"].T)
    W = x["W_down0"]
    outs = []
    for lo in range(0, T, w.C):
        hi = min(lo + w.C, T)
        outs.append(Z[lo:hi] @ W.T)
        W = W + w.eta * (V[lo:hi].T @ Z[lo:hi])
    (torch.cat(outs) * dO[0]).sum().backward()
    dV = V.grad.numpy()
    for c in range(w.d):
        M = np.zeros((T, T))  # Y[:, c] = M X0[:, c]
        for t in range(T):
            for s in range(k):
                src = t + 1 - (k - 1) + s
                if 0 <= src < T:
                    M[t, src] = cw[c, s].item()
        assert np.abs(M.T @ dV[:, c] - grads["X0"][0, :, c].numpy()).max() < 1e-10
