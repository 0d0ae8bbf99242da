"""Pins of the CPU oracle to things other than itself (CPU only).

Each test ties a part of oracle/oracle.py to something the pages or the
mathematics fix independently of the oracle's own code:
  * hand-derived worked examples (tests/golden/),
  * closed forms evaluated with library routines (torch fp64 silu / conv1d),
  * the 3-step prefix-sum form of the zhichai.net page (§3.2, Steps 1-3),
    computed by brute-force summation,
  * the linear-attention rearrangement of the state form,
  * linearity in eta, causality, batch independence,
  * a central finite-difference gradient of the printed loss (§3.3),
  * an independently written plain-C twin.
The last test plants plausible mistakes in copies of the oracle and checks
that the pins reject every one of them.
"""
import json
import os

import numpy as np
import pytest
import torch

from oracle import oracle
from oracle.twin import twin_layer_forward
from weight_mlp_layers_swiglu_b300.inputs import random_case

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _np(x):
    return oracle._f64(x)


def _rel(a, b):
    a, b = np.asarray(a), np.asarray(b)
    den = np.abs(b).max()
    return float(np.abs(a - b).max() / (den if den > 0 else 1.0))


def _case(B=1, T=37, d=6, f=10, C=8, k=3, eta=0.3, seed=11, dtype="f32"):
    w, x = random_case(B, T, d, f, C, k, eta, dtype, seed)
    return w, {n: _np(t) for n, t in x.items()}


def _run(x, C, eta, fwd=oracle.layer_forward):
    return fwd(x["H"], x["X0"], x["W_gate"], x["W_up"], x["W_down0"], x["W_target"], x["conv_w"], C, eta)


# --------------------------------------------------------------------------- golden


@pytest.mark.parametrize("name", ["hand_worked_T4_d2.json", "hand_worked_T3_ragged.json"])
def test_hand_worked_examples(name):
    g = json.load(open(os.path.join(GOLDEN, name)))
    a = {k: np.array(g[k], dtype=np.float64) for k in ("H", "W_gate", "W_up", "X0", "conv_w", "W_target", "W_down0")}
    tol = g["tolerance_rel"]
    Z = oracle.swiglu(a["H"], a["W_gate"], a["W_up"])
    assert _rel(Z, g["expected_Z"]) < tol
    V = oracle.target(a["X0"], a["conv_w"], a["W_target"])
    assert _rel(V, g["expected_V"]) < tol
    O, Wf = oracle.layer_forward(a["H"], a["X0"], a["W_gate"], a["W_up"], a["W_down0"], a["W_target"],
                                 a["conv_w"], g["C"], g["eta"])
    assert _rel(O[0], g["expected_O"]) < tol
    assert _rel(Wf[0], g["expected_W_final"]) < tol


# --------------------------------------------------------------------------- closed forms


def _torch_swiglu_mlp(x, W_down):
    """Plain gated MLP with torch's own SiLU and linear (fp64): the eta = 0 closed form."""
    H = torch.from_numpy(x["H"])
    Wg, Wu = torch.from_numpy(x["W_gate"]), torch.from_numpy(x["W_up"])
    Z = torch.nn.functional.silu(torch.nn.functional.linear(H, Wg)) * torch.nn.functional.linear(H, Wu)
    return torch.nn.functional.linear(Z, torch.from_numpy(W_down)).numpy(), Z.numpy()


def test_eta_zero_is_plain_swiglu_mlp():
    w, x = _case(B=2, T=40, C=8)
    O, Wf = _run(x, w.C, 0.0)
    O_ref, Z_ref = _torch_swiglu_mlp(x, x["W_down0"])
    assert _rel(O, O_ref) < 1e-12
    assert np.array_equal(Wf, np.broadcast_to(x["W_down0"], Wf.shape))
    assert _rel(oracle.swiglu(x["H"][0], x["W_gate"], x["W_up"]), Z_ref[0]) < 1e-12


def test_single_chunk_closed_form():
    w, x = _case(B=1, T=19, C=64)  # C >= T: one chunk
    O, Wf = _run(x, w.C, w.eta)
    O_ref, Z_ref = _torch_swiglu_mlp(x, x["W_down0"])
    assert _rel(O, O_ref) < 1e-12
    Y = torch.nn.functional.conv1d(torch.from_numpy(x["X0"][0]).T[None], torch.from_numpy(x["conv_w"])[:, None, :],
                                   padding=w.k - 1, groups=w.d)[0, :, : w.T].T.numpy()
    V = Y @ x["W_target"]
    assert _rel(Wf[0], x["W_down0"] + w.eta * V.T @ Z_ref[0]) < 1e-12


def test_conv_matches_torch_conv1d_and_impulse():
    rng = np.random.default_rng(3)
    T, d, k = 23, 5, 4
    X0 = rng.standard_normal((T, d))
    cw = rng.standard_normal((d, k))
    # torch's cross-correlation with k-1 zero padding on both sides, first T outputs = causal conv
    Y_t = torch.nn.functional.conv1d(torch.from_numpy(X0).T[None], torch.from_numpy(cw)[:, None, :],
                                     padding=k - 1, groups=d)[0, :, :T].T.numpy()
    assert _rel(oracle.causal_conv(X0, cw), Y_t) < 1e-14
    # impulse at t0 in channel c: Y[t0 + s, c] = conv_w[c, k-1-s] (tap k-1 is the current token)
    t0, c = 7, 2
    imp = np.zeros((T, d))
    imp[t0, c] = 1.0
    Y = oracle.causal_conv(imp, cw)
    for s in range(k):
        assert Y[t0 + s, c] == cw[c, k - 1 - s]
    assert np.count_nonzero(Y) == k
    assert np.all(Y[:t0] == 0)
    # k = 1 with unit weight is the identity; W_target = I gives V = Y
    assert np.array_equal(oracle.causal_conv(X0, np.ones((d, 1))), X0)
    assert np.array_equal(oracle.target(X0, np.ones((d, 1)), np.eye(d)), X0)


def test_conv_restarts_per_sequence():
    w, x = _case(B=2, T=12, C=4, k=4)
    V0 = oracle.target(x["X0"][1], x["conv_w"], x["W_target"])
    # sequence 1's first rows must not see sequence 0's last tokens
    Vcat = oracle.target(x["X0"].reshape(-1, w.d), x["conv_w"], x["W_target"])[w.T:]
    assert _rel(Vcat[w.k - 1:], V0[w.k - 1:]) < 1e-13
    assert not np.allclose(Vcat[:1], V0[:1])


# --------------------------------------------------------------------------- the 3-step form


def _brute_force_three_step(x, C, eta):
    """Steps 1-3 of the zhichai.net page §3.2: all Delta_i independently, an explicit
    exclusive prefix sum, then every chunk applied with its own weight."""
    H, X0 = x["H"][0], x["X0"][0]
    A = H @ x["W_gate"].T
    Z = A / (1.0 + np.exp(-A)) * (H @ x["W_up"].T)
    T, d = X0.shape
    k = x["conv_w"].shape[1]
    Y = np.zeros_like(X0)
    for t in range(T):
        for s in range(k):
            if t - k + 1 + s >= 0:
                Y[t] += x["conv_w"][:, s] * X0[t - k + 1 + s]
    V = Y @ x["W_target"]
    bounds = list(range(0, T, C)) + [T]
    deltas = [sum(np.outer(V[t], Z[t]) for t in range(bounds[i], bounds[i + 1])) for i in range(len(bounds) - 1)]
    O = np.zeros((T, d))
    for i in range(len(deltas)):
        W_i = x["W_down0"] + eta * sum((deltas[j] for j in range(i)), np.zeros_like(x["W_down0"]))
        for t in range(bounds[i], bounds[i + 1]):
            O[t] = W_i @ Z[t]
    W_fin = x["W_down0"] + eta * sum(deltas, np.zeros_like(x["W_down0"]))
    return O, W_fin


@pytest.mark.parametrize("T,C", [(32, 8), (37, 8), (8, 8), (1, 4)])
def test_sequential_loop_equals_prefix_sum_form(T, C):
    w, x = _case(T=T, C=C)
    O, Wf = _run(x, C, w.eta)
    O_b, W_b = _brute_force_three_step(x, C, w.eta)
    assert _rel(O[0], O_b) < 1e-12
    assert _rel(Wf[0], W_b) < 1e-12


def test_chunk_weights_and_apply_compose_to_the_layer():
    w, x = _case(T=45, C=8)
    Z = oracle.swiglu(x["H"][0], x["W_gate"], x["W_up"])
    V = oracle.target(x["X0"][0], x["conv_w"], x["W_target"])
    W_eff, W_fin = oracle.chunk_weights(V, Z, x["W_down0"], w.C, w.eta)
    assert W_eff.shape == (6, w.d, w.d_ff)
    assert np.array_equal(W_eff[0], x["W_down0"])
    O = oracle.chunk_apply(Z, W_eff, w.C)
    O_l, W_l = _run(x, w.C, w.eta)
    assert _rel(O, O_l[0]) < 1e-13 and _rel(W_fin, W_l[0]) < 1e-13


def test_linear_attention_identity():
    """O_i = Z_i W0^T + eta sum_{j<i} (Z_i Z_j^T) V_j, a rearrangement of the state form."""
    w, x = _case(T=50, C=8, eta=0.7)
    O, _ = _run(x, w.C, w.eta)
    Z = oracle.swiglu(x["H"][0], x["W_gate"], x["W_up"])
    V = oracle.target(x["X0"][0], x["conv_w"], x["W_target"])
    O_la = Z @ x["W_down0"].T
    for lo, hi in oracle.chunk_rows(w.T, w.C):
        if lo > 0:
            O_la[lo:hi] += w.eta * (Z[lo:hi] @ Z[:lo].T) @ V[:lo]
    assert _rel(O[0], O_la) < 1e-12


def test_linearity_in_eta():
    w, x = _case(B=2, T=33, C=8)
    O0, W0 = _run(x, w.C, 0.0)
    O1, W1 = _run(x, w.C, 1.0)
    for eta in (0.25, -1.5, 3.0):
        O, W = _run(x, w.C, eta)
        assert _rel(O, O0 + eta * (O1 - O0)) < 1e-12
        assert _rel(W, W0 + eta * (W1 - W0)) < 1e-12


# --------------------------------------------------------------------------- causality


def test_causality():
    w, x = _case(T=40, C=8, k=3)
    O, Wf = _run(x, w.C, w.eta)
    for i in (0, 2, 4):
        lo, hi = i * w.C, (i + 1) * w.C
        # X0 inside chunk i: chunks <= i unchanged (the target only feeds later chunks' weights)
        xp = dict(x)
        xp["X0"] = x["X0"].copy()
        xp["X0"][0, lo + 2] += 1.0
        Op, Wp = _run(xp, w.C, w.eta)
        assert np.array_equal(Op[0, :hi], O[0, :hi])
        if hi < w.T:
            assert not np.allclose(Op[0, hi:], O[0, hi:])
        assert not np.allclose(Wp, Wf)
        # H inside chunk i: chunks < i unchanged
        xp = dict(x)
        xp["H"] = x["H"].copy()
        xp["H"][0, lo + 3] += 1.0
        Op, _ = _run(xp, w.C, w.eta)
        assert np.array_equal(Op[0, :lo], O[0, :lo])
        assert not np.allclose(Op[0, lo:hi], O[0, lo:hi])
    # X0 in the last chunk: O unchanged, only the final state moves
    xp = dict(x)
    xp["X0"] = x["X0"].copy()
    xp["X0"][0, -1] += 1.0
    Op, Wp = _run(xp, w.C, w.eta)
    assert np.array_equal(Op, O)
    assert not np.allclose(Wp, Wf)


def test_batch_sequences_are_independent():
    w, x = _case(B=3, T=21, C=8)
    O, Wf = _run(x, w.C, w.eta)
    for b in range(3):
        xb = dict(x)
        xb["H"], xb["X0"] = x["H"][b:b + 1], x["X0"][b:b + 1]
        Ob, Wb = _run(xb, w.C, w.eta)
        assert np.array_equal(Ob[0], O[b]) and np.array_equal(Wb[0], Wf[b])


# --------------------------------------------------------------------------- gradient of the printed loss


def test_update_is_negative_gradient_of_loss():
    """Delta_i = V_i^T Z_i equals -dL_i/dW for L_i = -<V_i, Z_i W^T>_F (central differences)."""
    rng = np.random.default_rng(5)
    c, d, f = 4, 3, 5
    V = rng.standard_normal((c, d))
    Z = rng.standard_normal((c, f))
    W = rng.standard_normal((d, f))

    def loss(Wm):
        return -np.sum(V * (Z @ Wm.T))

    h = 1e-6
    G = np.zeros_like(W)
    for o in range(d):
        for j in range(f):
            E = np.zeros_like(W)
            E[o, j] = h
            G[o, j] = (loss(W + E) - loss(W - E)) / (2 * h)
    assert _rel(oracle.chunk_delta(V, Z), -G) < 1e-8


# --------------------------------------------------------------------------- independent twin


@pytest.mark.parametrize("B,T,d,f,C,k", [(1, 16, 4, 6, 4, 2), (2, 29, 5, 7, 8, 3), (1, 5, 3, 4, 8, 4), (1, 40, 8, 16, 16, 1)])
def test_plain_c_twin_agrees(B, T, d, f, C, k):
    w, x = _case(B=B, T=T, d=d, f=f, C=C, k=k, eta=0.2, seed=B * 100 + T)
    O, Wf = _run(x, C, w.eta)
    Ot, Wt = _run(x, C, w.eta, fwd=twin_layer_forward)
    assert _rel(O, Ot) < 1e-12 and _rel(Wf, Wt) < 1e-12


def test_bf16_inputs_are_widened_exactly():
    w, x = random_case(1, 12, 8, 16, 4, 4, 1.0 / 4, "bf16", 9)
    H = oracle._f64(x["H"])
    assert np.array_equal(H, x["H"].to(torch.float64).numpy())
    # bf16 values carry 8 significant bits: their fp32 widening is exact too
    assert np.array_equal(H, x["H"].float().double().numpy())


# --------------------------------------------------------------------------- the pins catch planted mistakes


def _mutant(kind):
    """A copy of the oracle's layer with one plausible mistake planted in it."""

    def fwd(H, X0, W_gate, W_up, W_down0, W_target, conv_w, C, eta):
        H, X0 = oracle._f64(H), oracle._f64(X0)
        Wg, Wu, W0, Wt, cw = (oracle._f64(a) for a in (W_gate, W_up, W_down0, W_target, conv_w))
        if kind == "taps_reversed":
            cw = cw[:, ::-1]
        if kind == "target_transposed":
            Wt = Wt.T
        if kind == "up_transposed_gate":
            Wg, Wu = Wu, Wg
        B, T, d = H.shape
        O = np.zeros((B, T, d))
        Wf = np.zeros((B, d, Wg.shape[0]))
        for b in range(B):
            A = H[b] @ Wg.T
            Z = (A / (1 + np.exp(-A)) if kind != "sigmoid_only" else 1 / (1 + np.exp(-A))) * (H[b] @ Wu.T)
            V = oracle.causal_conv(X0[b], cw) @ Wt
            W = W0.copy()
            for lo, hi in oracle.chunk_rows(T, C):
                step = eta * (V[lo:hi].T @ Z[lo:hi])
                if kind == "sign_flipped":
                    step = -step
                if kind == "inclusive":
                    W = W + step
                    O[b, lo:hi] = Z[lo:hi] @ W.T
                    continue
                O[b, lo:hi] = Z[lo:hi] @ W.T
                W = W + step
            Wf[b] = W
        return O, Wf

    return fwd


@pytest.mark.parametrize("kind", ["taps_reversed", "target_transposed", "up_transposed_gate", "sigmoid_only",
                                  "sign_flipped", "inclusive"])
def test_golden_pins_reject_planted_mistakes(kind):
    g = json.load(open(os.path.join(GOLDEN, "hand_worked_T4_d2.json")))
    a = {k: np.array(g[k], dtype=np.float64) for k in ("H", "W_gate", "W_up", "X0", "conv_w", "W_target", "W_down0")}
    O, Wf = _mutant(kind)(a["H"][None], a["X0"][None], a["W_gate"], a["W_up"], a["W_down0"], a["W_target"],
                          a["conv_w"], g["C"], g["eta"])
    ok = _rel(O[0], g["expected_O"]) < 1e-9 and _rel(Wf[0], g["expected_W_final"]) < 1e-9
    assert not ok, f"planted mistake {kind!r} passed the worked example"
    # the unmutated copy passes
    O, Wf = _mutant("none")(a["H"][None], a["X0"][None], a["W_gate"], a["W_up"], a["W_down0"], a["W_target"],
                            a["conv_w"], g["C"], g["eta"])
    assert _rel(O[0], g["expected_O"]) < 1e-12 and _rel(Wf[0], g["expected_W_final"]) < 1e-12
