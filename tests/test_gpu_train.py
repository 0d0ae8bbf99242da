"""The training pair of entries: ipttt_layer_forward_train (the layer plus the activations the
backward pass reads) and ipttt_layer_backward_saved (the backward half from them).

The forward must equal ipttt_layer_forward bit for bit, and the gradients must equal those of
ipttt_layer_backward (which recomputes the same activations with the same kernels) bit for
bit; ipttt_layer_backward is itself held to the gradient oracle in test_gpu_backward.py, and
the saved path is checked against the oracle here too."""
import pytest
import torch

from oracle.oracle_grad import layer_backward
from tests.util import TOL, rel_err, seeded, to_dev
from weight_mlp_layers_swiglu_b300.inputs import random_case

pytestmark = pytest.mark.gpu

GRADS = ["H", "X0", "W_gate", "W_up", "W_down0", "W_target", "conv_w"]


@pytest.fixture(scope="module")
def ctx():
    import weight_mlp_layers_swiglu_b300 as pkg

    c = pkg.Context(0)
    yield c
    c.close()


def _inputs(dt, B, T, d, f, C, k, seed, no_proj=False):
    w, x = random_case(B, T, d, f, C, k, 2.0 / C, dt, seed)
    if no_proj:
        x["W_target"] = None
    xd = {n: (None if v is None else v.cuda().contiguous()) for n, v in x.items()}
    tdt = x["H"].dtype
    dO = seeded((B, T, d), 1.0, tdt, seed + 1, "cuda")
    dWf = seeded((B, d, f), 0.5, torch.float32, seed + 2, "cuda")
    return w, x, xd, dO, dWf


@pytest.mark.parametrize("no_proj", [False, True])
@pytest.mark.parametrize("dt,B,T,d,f,C,k", [
    ("bf16", 2, 700, 256, 512, 256, 4),    # fused pair kernel
    ("bf16", 1, 300, 192, 384, 128, 3),    # single-CTA fused kernel (C % 256 != 0), ragged tails
    ("f32", 2, 200, 64, 128, 48, 4),
])
def test_train_pair_matches_forward_and_backward(ctx, no_proj, dt, B, T, d, f, C, k):
    w, x, xd, dO, dWf = _inputs(dt, B, T, d, f, C, k, 300 + T, no_proj)
    args = (xd["H"], xd["X0"], xd["W_gate"], xd["W_up"], xd["W_down0"], xd["W_target"], xd["conv_w"], C, w.eta)
    O_ref, W_ref = (t.clone() for t in ctx.layer_forward(*args))
    g_ref = ctx.layer_backward(*args, dO, dWf)
    O, Wf, saved = ctx.layer_forward_train(*args)
    g = ctx.layer_backward_saved(xd["H"], xd["X0"], xd["W_gate"], xd["W_up"], xd["W_target"], xd["conv_w"], C, w.eta,
                                 saved, dO, dWf)
    assert ctx.sync() == 0, ctx.last_error()
    assert torch.equal(O, O_ref) and torch.equal(Wf, W_ref)
    for n in GRADS:
        if g_ref[n] is None:
            assert g[n] is None
        else:
            assert torch.equal(g[n], g_ref[n]), n
    ref = layer_backward(x["H"], x["X0"], x["W_gate"], x["W_up"], x["W_down0"], x["W_target"], x["conv_w"], C, w.eta,
                         dO.cpu(), dWf.cpu())
    for n in GRADS:
        if ref[n] is not None:
            assert rel_err(g[n], ref[n]) <= TOL[dt], n


def test_train_shifted_window(ctx):
    w, x, xd, dO, dWf = _inputs("bf16", 2, 512, 128, 256, 256, 3, 51)
    args = (xd["H"], xd["X0"], xd["W_gate"], xd["W_up"], xd["W_down0"], xd["W_target"], xd["conv_w"], 256, w.eta)
    ctx.set_target_shift(1)
    try:
        g_ref = ctx.layer_backward(*args, dO, dWf)
        _, _, saved = ctx.layer_forward_train(*args)
        g = ctx.layer_backward_saved(xd["H"], xd["X0"], xd["W_gate"], xd["W_up"], xd["W_target"], xd["conv_w"], 256,
                                     w.eta, saved, dO, dWf)
        assert ctx.sync() == 0, ctx.last_error()
    finally:
        ctx.set_target_shift(0)
    for n in GRADS:
        assert torch.equal(g[n], g_ref[n]), n


def test_train_rejects_small_saved_buffer(ctx):
    import weight_mlp_layers_swiglu_b300 as pkg

    w, x, xd, dO, dWf = _inputs("bf16", 1, 256, 128, 256, 128, 4, 52)
    small = torch.empty(4096, dtype=torch.uint8, device="cuda")
    with pytest.raises(pkg.IptttError) as e:
        ctx.layer_forward_train(xd["H"], xd["X0"], xd["W_gate"], xd["W_up"], xd["W_down0"], xd["W_target"],
                                xd["conv_w"], 128, w.eta, saved=small)
    assert e.value.status == 3
    with pytest.raises(pkg.IptttError) as e:
        ctx.layer_backward_saved(xd["H"], xd["X0"], xd["W_gate"], xd["W_up"], xd["W_target"], xd["conv_w"], 128,
                                 w.eta, small, dO, dWf)
    assert e.value.status == 3
