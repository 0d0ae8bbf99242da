"""Pins of the oracle's ablation variants (CPU only), the axes of the zhichai.net page's §6
ablation table: without the projection (W_target = I), without the convolution (k = 1, unit
tap), both, and the target window that ends at the next token."""
import numpy as np
import torch

from oracle import oracle
from weight_mlp_layers_swiglu_b300.inputs import random_case


def _rel(a, b):
    den = np.abs(b).max()
    return float(np.abs(a - b).max() / (den if den else 1.0))


def _x(T=30, d=6, f=10, C=8, k=3, seed=31):
    w, x = random_case(1, T, d, f, C, k, 0.5, "f32", seed)
    return w, {n: oracle._f64(t) for n, t in x.items()}


def test_no_projection_equals_identity_projection():
    w, x = _x()
    O1, W1 = oracle.layer_forward(x["H"], x["X0"], x["W_gate"], x["W_up"], x["W_down0"], None, x["conv_w"], w.C, w.eta)
    O2, W2 = oracle.layer_forward(x["H"], x["X0"], x["W_gate"], x["W_up"], x["W_down0"], np.eye(w.d), x["conv_w"],
                                  w.C, w.eta)
    assert np.array_equal(O1, O2) and np.array_equal(W1, W2)


def test_no_conv_no_projection_is_the_embedding_target():
    w, x = _x(k=1)
    V = oracle.target(x["X0"][0], np.ones((w.d, 1)), None)
    assert np.array_equal(V, x["X0"][0])


def test_next_token_window_is_the_causal_window_one_token_later():
    """shift = 1 at token t equals the causal conv at t + 1 of X0 with a zero row appended,
    checked against torch's conv1d."""
    rng = np.random.default_rng(8)
    T, d, k = 17, 4, 3
    X0 = rng.standard_normal((T, d))
    cw = rng.standard_normal((d, k))
    Xz = np.concatenate([X0, np.zeros((1, d))])
    Y_t = torch.nn.functional.conv1d(torch.from_numpy(Xz).T[None], torch.from_numpy(cw)[:, None, :],
                                     padding=k - 1, groups=d)[0, :, : T + 1].T.numpy()
    assert _rel(oracle.causal_conv(X0, cw, shift=1), Y_t[1:]) < 1e-14
    # the shifted target reads the next token: an impulse at t0 reaches Y[t0 - 1]
    imp = np.zeros((T, d))
    imp[5, 1] = 1.0
    Y = oracle.causal_conv(imp, cw, shift=1)
    assert Y[4, 1] == cw[1, k - 1] and np.all(Y[:4] == 0)


def test_next_token_window_layer_still_uses_earlier_chunks_only():
    """With shift = 1 the chunk-i update reads X0 up to the first token of chunk i+1, so O of
    chunk i+1 depends on that token (but O of chunks <= i does not)."""
    w, x = _x(T=32, C=8)
    O, _ = oracle.layer_forward(x["H"], x["X0"], x["W_gate"], x["W_up"], x["W_down0"], x["W_target"], x["conv_w"],
                                w.C, w.eta, shift=1)
    xp = dict(x)
    xp["X0"] = x["X0"].copy()
    xp["X0"][0, 16] += 1.0  # first token of chunk 2
    Op, _ = oracle.layer_forward(xp["H"], xp["X0"], x["W_gate"], x["W_up"], x["W_down0"], x["W_target"], x["conv_w"],
                                 w.C, w.eta, shift=1)
    assert np.array_equal(Op[0, :16], O[0, :16])
    assert not np.allclose(Op[0, 16:24], O[0, 16:24])
