"""Pins of the oracle's resumable layer (CPU only).

The resumable call is pinned against the single-call layer, which is itself pinned by
tests/test_oracle_pins.py: a sequence cut at any multiple of C and run as several calls,
each continuing from the previous call's fp64 state and conv halo, must give the single call's
outputs; a first call (zero halo, W_down0 as the state) must be the plain layer; the halo is
what the causal convolution would have read.
"""
import numpy as np
import pytest
import torch

from oracle import oracle
from weight_mlp_layers_swiglu_b300.inputs import random_case


def _rel(a, b):
    den = np.abs(b).max()
    return float(np.abs(a - b).max() / (den if den else 1.0))


def _case(B=2, T=40, d=6, f=10, C=8, k=3, eta=0.4, seed=21):
    w, x = random_case(B, T, d, f, C, k, eta, "f32", seed)
    return w, {n: oracle._f64(t) for n, t in x.items()}


def _resume(x, H, X0, W_state, halo, C, eta):
    return oracle.layer_resume(H, X0, x["W_gate"], x["W_up"], x["W_target"], x["conv_w"], W_state, halo, C, eta)


@pytest.mark.parametrize("cuts", [[16], [8, 24], [8, 16, 24, 32], [40]])
def test_split_at_chunk_multiples_equals_one_call(cuts):
    w, x = _case()
    O_ref, W_ref = oracle.layer_forward(x["H"], x["X0"], x["W_gate"], x["W_up"], x["W_down0"], x["W_target"],
                                        x["conv_w"], w.C, w.eta)
    state = np.broadcast_to(x["W_down0"], (w.B, w.d, w.d_ff)).copy()
    halo = np.zeros((w.B, w.k - 1, w.d))
    outs = []
    for lo, hi in zip([0] + cuts, cuts + [w.T]):
        if hi <= lo:
            continue
        O, state, halo = _resume(x, x["H"][:, lo:hi], x["X0"][:, lo:hi], state, halo, w.C, w.eta)
        outs.append(O)
    assert _rel(np.concatenate(outs, axis=1), O_ref) < 1e-12
    assert _rel(state, W_ref) < 1e-12


def test_first_call_is_the_plain_layer_and_halo_is_the_tail():
    w, x = _case(T=13, k=4)
    state = np.broadcast_to(x["W_down0"], (w.B, w.d, w.d_ff)).copy()
    O, Wf, halo = _resume(x, x["H"], x["X0"], state, np.zeros((w.B, w.k - 1, w.d)), w.C, w.eta)
    O_ref, W_ref = oracle.layer_forward(x["H"], x["X0"], x["W_gate"], x["W_up"], x["W_down0"], x["W_target"],
                                        x["conv_w"], w.C, w.eta)
    assert np.array_equal(O, O_ref) and np.array_equal(Wf, W_ref)
    assert np.array_equal(halo, x["X0"][:, -(w.k - 1):])
    # a call shorter than the halo keeps the older halo rows in front
    h0 = np.arange(w.B * (w.k - 1) * w.d, dtype=float).reshape(w.B, w.k - 1, w.d)
    _, _, h1 = _resume(x, x["H"][:, :1], x["X0"][:, :1], state, h0, w.C, w.eta)
    assert np.array_equal(h1[:, :-1], h0[:, 1:]) and np.array_equal(h1[:, -1], x["X0"][:, 0])


def test_halo_matches_torch_conv_on_the_joined_sequence():
    rng = np.random.default_rng(4)
    T, d, k = 9, 5, 4
    X = rng.standard_normal((T + 6, d))
    cw = rng.standard_normal((d, k))
    Y_all = torch.nn.functional.conv1d(torch.from_numpy(X).T[None], torch.from_numpy(cw)[:, None, :],
                                       padding=k - 1, groups=d)[0, :, : T + 6].T.numpy()
    Y = oracle.causal_conv(X[6:], cw, halo=X[6 - (k - 1): 6])
    assert _rel(Y, Y_all[6:]) < 1e-14


def test_state_carries_learning_between_calls():
    """With eta != 0 the second call's outputs depend on the first call's tokens only
    through the carried state and halo."""
    w, x = _case(T=32)
    state = np.broadcast_to(x["W_down0"], (w.B, w.d, w.d_ff)).copy()
    halo = np.zeros((w.B, w.k - 1, w.d))
    _, s1, h1 = _resume(x, x["H"][:, :16], x["X0"][:, :16], state, halo, w.C, w.eta)
    O2, _, _ = _resume(x, x["H"][:, 16:], x["X0"][:, 16:], s1, h1, w.C, w.eta)
    O2_fresh, _, _ = _resume(x, x["H"][:, 16:], x["X0"][:, 16:], state, halo, w.C, w.eta)
    assert not np.allclose(O2, O2_fresh)
