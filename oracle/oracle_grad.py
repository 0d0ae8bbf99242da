"""Gradients of the fast-weight SwiGLU layer: float64 autograd on the CPU.

TEST INFRASTRUCTURE ONLY (see oracle/oracle.py).  The layer is restated with plain torch
float64 ops -- the same literal chunk loop as oracle.sequence_forward (zhichai.net "In-Place
TTT：给LLM装上"临时记忆插槽"，让它边读边学", §3.1 gated MLP, §3.2 chunk loop, §3.3 target and
update rule) -- and torch's reverse-mode autodiff (a library step) differentiates it.  The
pages give no gradient formulas; they train models with the layer in place (continued and
from-scratch pretraining, page §5), which needs exactly these gradients: of
<dO, O> + <dW_final, W_final> with respect to every input, through the fast-weight chain.

Pinned in tests/test_oracle_grad.py by the forward's agreement with oracle.layer_forward and
by central finite differences along random directions, which do not use autodiff.
"""
from __future__ import annotations

import torch


def _t(x):
    if isinstance(x, torch.Tensor):
        return x.detach().to(torch.float64).clone()
    return torch.as_tensor(x, dtype=torch.float64).clone()


def forward_torch(H, X0, W_gate, W_up, W_down0, W_target, conv_w, C: int, eta: float, shift: int = 0):
    """O [B, T, d] and final W_down [B, d, d_ff], torch float64, differentiable.

    W_target None is the identity projection and shift = 1 the conv window ending at the next
    token (the ablation variants of the zhichai page's §6 table and its Theorem 1), as in
    oracle.target."""
    B, T, d = H.shape
    k = conv_w.shape[1]
    A = H @ W_gate.T
    Z = A * torch.sigmoid(A) * (H @ W_up.T)
    Xp = torch.cat([torch.zeros(B, k - 1, d, dtype=H.dtype), X0, torch.zeros(B, shift, d, dtype=H.dtype)], dim=1)
    Y = sum(conv_w[:, s] * Xp[:, s + shift: s + shift + T] for s in range(k))
    V = Y if W_target is None else Y @ W_target
    outs, finals = [], []
    for b in range(B):
        W = W_down0
        Ob = []
        for lo in range(0, T, C):
            hi = min(lo + C, T)
            Ob.append(Z[b, lo:hi] @ W.T)
            W = W + eta * (V[b, lo:hi].T @ Z[b, lo:hi])
        outs.append(torch.cat(Ob) if Ob else torch.zeros(0, d, dtype=H.dtype))
        finals.append(W)
    return torch.stack(outs), torch.stack(finals)


def layer_backward(H, X0, W_gate, W_up, W_down0, W_target, conv_w, C: int, eta: float, dO, dW_final=None,
                   shift: int = 0):
    """Gradients of <dO, O> + <dW_final, W_final> (dW_final None = 0) with respect to
    H, X0, W_gate, W_up, W_down0, W_target, conv_w, as a dict of float64 tensors (W_target's
    entry is None when W_target is None)."""
    names = ["H", "X0", "W_gate", "W_up", "W_down0", "W_target", "conv_w"]
    vals = (H, X0, W_gate, W_up, W_down0, W_target, conv_w)
    leaves = {n: (None if v is None else _t(v).requires_grad_(True)) for n, v in zip(names, vals)}
    O, Wf = forward_torch(*(leaves[n] for n in names), C, eta, shift)
    loss = (O * _t(dO)).sum()
    if dW_final is not None:
        loss = loss + (Wf * _t(dW_final)).sum()
    loss.backward()
    return {n: (None if leaves[n] is None else leaves[n].grad.detach()) for n in names}
