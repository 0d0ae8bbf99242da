"""The layer's backward pass on the GPU (ipttt_layer_backward through the C ABI) against the
gradient oracle (float64 autograd of the literal chunk loop on the CPU).

Every gradient is compared with the parity metric max|x - ref| / max|ref|.  fp32 runs on CUDA
cores with fp32 intermediates: 1e-4.  bf16 rounds each stored intermediate (Z, V, W_i, R_i,
dZ, dA, dU, dV, dY) to bf16 (relative 2^-9 each) and accumulates every product in fp32; the
errors of a few roundings in series stay well under 2e-2."""
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


def _run(ctx, dt, B, T, d, f, C, k, eta, seed, with_dWf=True, no_proj=False, shift=0):
    w, x = random_case(B, T, d, f, C, k, eta, dt, seed)
    if no_proj:
        x["W_target"] = None
    tdt = x["H"].dtype
    dO = seeded((B, T, d), 1.0, tdt, seed + 1)
    dWf = seeded((B, d, f), 0.5, torch.float32, seed + 2) if with_dWf else None
    xd = {n: (None if v is None else v.cuda().contiguous()) for n, v in x.items()}
    ctx.set_target_shift(shift)
    try:
        g = ctx.layer_backward(xd["H"], xd["X0"], xd["W_gate"], xd["W_up"], xd["W_down0"], xd["W_target"],
                               xd["conv_w"], C, eta, dO.cuda(), None if dWf is None else dWf.cuda())
        assert ctx.sync() == 0, ctx.last_error()
    finally:
        ctx.set_target_shift(0)
    ref = layer_backward(x["H"], x["X0"], x["W_gate"], x["W_up"], x["W_down0"], x["W_target"], x["conv_w"], C,
                         eta, dO, dWf, shift=shift)
    return g, ref


def _check(g, ref, tol):
    errs = {}
    for n in GRADS:
        if ref[n] is None:
            assert g[n] is None
            continue
        assert g[n].shape == ref[n].shape, n
        assert torch.isfinite(g[n].float()).all(), n
        errs[n] = rel_err(g[n], ref[n])
    print({n: f"{e:.2e}" for n, e in errs.items()})
    bad = {n: e for n, e in errs.items() if not e <= tol}
    assert not bad, f"gradients past {tol}: {bad} (all: {errs})"
    return errs


@pytest.mark.parametrize("dt,B,T,d,f,C,k", [
    ("bf16", 2, 640, 256, 512, 128, 4),
    ("bf16", 1, 300, 192, 384, 128, 3),    # ragged last chunk, tiles and K blocks
    ("bf16", 3, 130, 136, 264, 256, 2),    # one short chunk per sequence, d and d_ff off the tile grid
    ("f32", 2, 200, 64, 128, 48, 4),
    ("f32", 1, 77, 40, 56, 16, 1),
])
def test_backward_matches_oracle(ctx, dt, B, T, d, f, C, k):
    g, ref = _run(ctx, dt, B, T, d, f, C, k, 2.0 / C, 900 + T)
    _check(g, ref, TOL[dt])


@pytest.mark.parametrize("dt", ["bf16", "f32"])
def test_backward_without_final_state_gradient(ctx, dt):
    C = 128
    g, ref = _run(ctx, dt, 2, 384, 128, 256, C, 4, 2.0 / C, 41, with_dWf=False)
    _check(g, ref, TOL[dt])


@pytest.mark.parametrize("dt", ["bf16", "f32"])
def test_backward_identity_projection(ctx, dt):
    C = 128
    g, ref = _run(ctx, dt, 2, 256, 128, 256, C, 4, 2.0 / C, 42, no_proj=True)
    assert g["W_target"] is None
    _check(g, ref, TOL[dt])


@pytest.mark.parametrize("dt", ["bf16", "f32"])
def test_backward_shifted_target_window(ctx, dt):
    C = 128
    g, ref = _run(ctx, dt, 2, 300, 128, 256, C, 3, 2.0 / C, 43, shift=1)
    _check(g, ref, TOL[dt])


def test_backward_weight_gradient_sees_every_chunk(ctx):
    """dW_down0 sums the chunk gradients of every sequence: a scan that dropped or double-counted
    a chunk would move it by a whole chunk's share, far past the bound."""
    C = 128
    g, ref = _run(ctx, "bf16", 3, 1024, 128, 256, C, 4, 2.0 / C, 44)
    errs = _check(g, ref, TOL["bf16"])
    assert errs["W_down0"] <= 5e-3


def test_backward_no_tokens(ctx):
    """T = 0: every gradient is zero except dW_down0 = sum_b dW_final[b]."""
    B, d, f, k = 3, 64, 128, 4
    w, x = random_case(B, 0, d, f, 128, k, 0.1, "bf16", 5)
    xd = to_dev(x)
    dWf = seeded((B, d, f), 1.0, torch.float32, 6, "cuda")
    dO = torch.zeros((B, 0, d), dtype=torch.bfloat16, device="cuda")
    g = ctx.layer_backward(xd["H"], xd["X0"], xd["W_gate"], xd["W_up"], xd["W_down0"], xd["W_target"], xd["conv_w"],
                           128, 0.1, dO, dWf)
    assert ctx.sync() == 0
    for n in ["W_gate", "W_up", "W_target", "conv_w"]:
        assert torch.count_nonzero(g[n]) == 0, n
    assert torch.allclose(g["W_down0"], dWf.sum(0), rtol=1e-6, atol=1e-6)
    assert g["H"].numel() == 0 and g["X0"].numel() == 0


def test_backward_rejects_small_workspace_and_overlap(ctx):
    import weight_mlp_layers_swiglu_b300 as pkg

    w, x = random_case(1, 256, 128, 256, 128, 4, 0.1, "bf16", 7)
    xd = to_dev(x)
    dO = torch.zeros((1, 256, 128), dtype=torch.bfloat16, device="cuda")
    small = torch.empty(1024, dtype=torch.uint8, device="cuda")
    with pytest.raises(pkg.IptttError) as e:
        ctx.layer_backward(xd["H"], xd["X0"], xd["W_gate"], xd["W_up"], xd["W_down0"], xd["W_target"],
                           xd["conv_w"], 128, 0.1, dO, workspace=small)
    assert e.value.status == 3
    # dO doubling as the workspace overlaps an input
    n = pkg.backward_workspace_size(1, 256, 128, 256, 128, 4, pkg.BF16)
    big = torch.empty(n + 256 * 128 * 2, dtype=torch.uint8, device="cuda")
    dO_alias = big[:256 * 128 * 2].view(torch.bfloat16).view(1, 256, 128)
    with pytest.raises(pkg.IptttError) as e:
        ctx.layer_backward(xd["H"], xd["X0"], xd["W_gate"], xd["W_up"], xd["W_down0"], xd["W_target"],
                           xd["conv_w"], 128, 0.1, dO_alias, workspace=big)
    assert e.value.status == 1


@pytest.mark.slow
@pytest.mark.parametrize("name,T", [("small_0p4b", None), ("qwen3_4b_32k", 4096), ("serve_8x8k", 1024)])
def test_backward_at_workload_widths(ctx, name, T):
    """The bf16 workloads' own shapes (the 0.4B-scale layer at its full 32k tokens; the 4B-shaped
    layers at their full widths over a shorter prefix, which the float64 autograd oracle finishes
    in seconds) against the oracle, every gradient element by element."""
    import json
    import os

    from weight_mlp_layers_swiglu_b300.inputs import WORKLOADS, make_inputs

    w = WORKLOADS[name]
    if T is not None:
        w = w.with_(T=T)
    x = make_inputs(w)
    dO = seeded((w.B, w.T, w.d), 1.0, torch.bfloat16, 77)
    dWf = seeded((w.B, w.d, w.d_ff), 0.05, torch.float32, 78)
    xd = to_dev(x)
    g = ctx.layer_backward(xd["H"], xd["X0"], xd["W_gate"], xd["W_up"], xd["W_down0"], xd["W_target"],
                           xd["conv_w"], w.C, w.eta, dO.cuda(), dWf.cuda())
    assert ctx.sync() == 0, ctx.last_error()
    g = {n: (None if v is None else v.cpu()) for n, v in g.items()}
    del xd
    torch.cuda.empty_cache()
    ref = layer_backward(x["H"], x["X0"], x["W_gate"], x["W_up"], x["W_down0"], x["W_target"], x["conv_w"], w.C,
                         w.eta, dO, dWf)
    errs = _check(g, ref, TOL["bf16"])
    out = os.environ.get("IPTTT_RESULTS_DIR")  # optional: a directory for the measured errors
    if out and os.path.isdir(out):
        with open(os.path.join(out, f"parity_backward_{name}_T{w.T}.json"), "w") as f:
            json.dump({"workload": name, "T": w.T, **errs}, f)
    print(name, w.T, errs)
