"""Ablation variants of the target on the GPU against the oracle (the axes of the zhichai.net
page's §6 table): without the projection (W_target = NULL), without the convolution (k = 1,
unit tap), both, and the target window that ends at the next token."""
import pytest
import torch

from tests.util import layer_check, to_dev
from weight_mlp_layers_swiglu_b300.inputs import random_case

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ctx():
    import weight_mlp_layers_swiglu_b300 as pkg

    c = pkg.Context(0)
    yield c
    c.close()


def _run(ctx, w, x, W_target="given", shift=0, fused=True):
    xd = to_dev(x)
    Wt = xd["W_target"] if W_target == "given" else None
    ctx.set_target_shift(shift)
    ctx.set_fused_tail(fused)
    try:
        O, Wf = ctx.layer_forward(xd["H"], xd["X0"], xd["W_gate"], xd["W_up"], xd["W_down0"], Wt, xd["conv_w"],
                                  w.C, w.eta)
        assert ctx.sync() == 0, ctx.last_error()
    finally:
        ctx.set_target_shift(0)
        ctx.set_fused_tail(True)
    return O, Wf


@pytest.mark.parametrize("dt", ["bf16", "f32"])
@pytest.mark.parametrize("fused", [True, False])
def test_without_projection(ctx, dt, fused):
    w, x = random_case(2, 640, 256, 512, 128, 4, 4.0 / 128, dt, 61)
    O, Wf = _run(ctx, w, x, W_target=None, fused=fused)
    xi = dict(x)
    xi["W_target"] = torch.eye(w.d, dtype=x["W_target"].dtype)
    layer_check(w, xi, O, Wf)


@pytest.mark.parametrize("dt", ["bf16", "f32"])
def test_without_conv_and_projection(ctx, dt):
    w, x = random_case(1, 512, 256, 512, 128, 1, 4.0 / 128, dt, 62)
    x["conv_w"] = torch.ones_like(x["conv_w"])
    O, Wf = _run(ctx, w, x, W_target=None)
    xi = dict(x)
    xi["W_target"] = torch.eye(w.d, dtype=x["W_target"].dtype)
    layer_check(w, xi, O, Wf)


@pytest.mark.parametrize("dt", ["bf16", "f32"])
def test_next_token_window(ctx, dt):
    from oracle import oracle
    from tests.util import TOL, rel_err

    w, x = random_case(2, 640, 256, 512, 128, 4, 4.0 / 128, dt, 63)
    O, Wf = _run(ctx, w, x, shift=1)
    O_ref, W_ref = oracle.layer_forward(x["H"], x["X0"], x["W_gate"], x["W_up"], x["W_down0"], x["W_target"],
                                        x["conv_w"], w.C, w.eta, shift=1)
    assert rel_err(O, O_ref) <= TOL[dt] and rel_err(Wf, W_ref) <= TOL[dt]
    # and it differs from the causal window
    O0, _ = _run(ctx, w, x, shift=0)
    assert not torch.equal(O0, O)


def test_target_step_without_projection(ctx):
    from oracle import oracle
    from tests.util import rel_err, seeded

    X0 = seeded((2, 200, 256), 0.02, torch.bfloat16, 4, "cuda")
    cw = seeded((256, 4), 0.5, torch.bfloat16, 5, "cuda")
    V = torch.empty_like(X0)
    import ctypes

    st = ctx.lib.ipttt_target(ctx.h, ctypes.c_void_p(X0.data_ptr()), ctypes.c_void_p(cw.data_ptr()), None, 2, 200,
                              256, 4, 0.5, 1, None, ctypes.c_void_p(V.data_ptr()))
    assert st == 0 and ctx.sync() == 0
    for b in range(2):
        assert rel_err(V[b], 0.5 * oracle.causal_conv(X0[b].cpu(), cw.cpu())) <= 1e-2


def test_next_token_window_refused_by_piecewise_entry_points(ctx):
    """The shifted window's last target of a piece reads the next piece's first X0 row, which a
    piecewise call does not have: resumed calls, layer_totals and a host-buffer call that spans
    several pieces refuse it (UNSUPPORTED) and launch nothing, while a host-buffer call of one
    piece is one whole call and matches ipttt_layer_forward bit for bit."""
    import weight_mlp_layers_swiglu_b300 as pkg

    w, x = random_case(1, 512, 256, 512, 128, 4, 4.0 / 128, "bf16", 64)
    xd = to_dev(x)
    B, T, d, f, k = w.B, w.T, w.d, w.d_ff, w.k
    W_state = xd["W_down0"].float()[None].repeat(B, 1, 1).contiguous()
    ctx.set_target_shift(1)
    try:
        with pytest.raises(pkg.IptttError) as e:
            ctx.layer_resume(xd["H"], xd["X0"], xd["W_gate"], xd["W_up"], xd["W_target"], xd["conv_w"], W_state,
                             None, w.C, w.eta)
        assert e.value.status == 2  # IPTTT_ERR_UNSUPPORTED
        with pytest.raises(pkg.IptttError) as e:
            ctx.layer_totals(xd["H"], xd["X0"], xd["W_gate"], xd["W_up"], xd["W_target"], xd["conv_w"], None, w.C,
                             w.eta)
        assert e.value.status == 2
        # one piece: the whole call
        O_pin = torch.empty((B, T, d), dtype=torch.bfloat16).pin_memory()
        W_pin = torch.empty((B, d, f), dtype=torch.float32).pin_memory()
        ctx.layer_forward_host(x["H"].pin_memory(), x["X0"].pin_memory(), xd["W_gate"], xd["W_up"], xd["W_down0"],
                               xd["W_target"], xd["conv_w"], w.C, w.eta, O_pin, W_pin)
        assert ctx.sync() == 0, ctx.last_error()
        O, Wf = ctx.layer_forward(xd["H"], xd["X0"], xd["W_gate"], xd["W_up"], xd["W_down0"], xd["W_target"],
                                  xd["conv_w"], w.C, w.eta)
        assert ctx.sync() == 0
        assert torch.equal(O_pin, O.cpu()) and torch.equal(W_pin, Wf.cpu())
        # several pieces: refused
        wl, xl = random_case(1, 8192, 128, 256, 128, 4, 1.0 / 128, "bf16", 65)
        xld = to_dev(xl)
        Ol = torch.empty((1, 8192, 128), dtype=torch.bfloat16).pin_memory()
        Wl = torch.empty((1, 128, 256), dtype=torch.float32).pin_memory()
        with pytest.raises(pkg.IptttError) as e:
            ctx.layer_forward_host(xl["H"].pin_memory(), xl["X0"].pin_memory(), xld["W_gate"], xld["W_up"],
                                   xld["W_down0"], xld["W_target"], xld["conv_w"], wl.C, wl.eta, Ol, Wl)
        assert e.value.status == 2
    finally:
        ctx.set_target_shift(0)
    assert ctx.sync() == 0
