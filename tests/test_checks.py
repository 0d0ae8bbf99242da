"""The parity checker used by the GPU tests, exercised on the CPU: outputs with a planted
mistake (made by a mutated copy of the oracle's chunk loop) must fail it, and the oracle's
own outputs rounded to bf16 must pass it."""
import numpy as np
import pytest
import torch

from oracle import oracle
from tests.util import _bf16, layer_check
from weight_mlp_layers_swiglu_b300.inputs import random_case


def _planted(x, C, eta, kind):
    """A copy of the oracle's chunk loop with one planted mistake."""
    O, Wf = [], []
    for b in range(x["H"].shape[0]):
        Z = oracle.swiglu(x["H"][b], x["W_gate"], x["W_up"])
        V = oracle.target(x["X0"][b], x["conv_w"], x["W_target"])
        W = oracle._f64(x["W_down0"]).copy()
        Ob = np.zeros((Z.shape[0], W.shape[0]))
        rows = oracle.chunk_rows(Z.shape[0], C)
        for i, (lo, hi) in enumerate(rows):
            step = eta * V[lo:hi].T @ Z[lo:hi]
            if kind == "inclusive":
                W = W + step
                Ob[lo:hi] = Z[lo:hi] @ W.T
                continue
            Ob[lo:hi] = Z[lo:hi] @ W.T
            if kind == "drop_chunk" and i == 1:
                continue
            if kind == "lagged" and i > 0:  # each chunk uses the weight two updates back
                Ob[lo:hi] = Z[lo:hi] @ (W - eta * V[rows[i - 1][0]:rows[i - 1][1]].T @ Z[rows[i - 1][0]:rows[i - 1][1]]).T
            W = W + step
        O.append(Ob)
        Wf.append(W)
    return np.stack(O), np.stack(Wf)


CASE = (1, 1024, 256, 512, 128, 4, 4.0 / 128, "bf16", 123)


def test_checker_accepts_bf16_rounded_oracle_outputs():
    w, x = random_case(*CASE)
    O, Wf = oracle.layer_forward(x["H"], x["X0"], x["W_gate"], x["W_up"], x["W_down0"], x["W_target"],
                                 x["conv_w"], w.C, w.eta)
    errs = layer_check(w, x, _bf16(O), Wf.astype(np.float32).astype(np.float64))
    assert errs["O"] < 1e-2


@pytest.mark.parametrize("kind", ["inclusive", "drop_chunk", "lagged"])
def test_checker_rejects_planted_mistakes(kind):
    w, x = random_case(*CASE)
    O, Wf = _planted(x, w.C, w.eta, kind)
    with pytest.raises(AssertionError):
        layer_check(w, x, _bf16(O), Wf)
