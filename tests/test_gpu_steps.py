"""Per-kernel parity on the GPU: each step of the layer, called through the C ABI, against the
oracle's function for the same step on the same (bf16 or fp32) inputs.  Shapes span several
tiles and end in ragged tails (rows, d, d_ff and the last chunk)."""
import numpy as np
import pytest
import torch

from oracle import oracle
from tests.util import rel_err, seeded

pytestmark = pytest.mark.gpu

DT = {"bf16": torch.bfloat16, "f32": torch.float32}
# Each step's own bound: bf16 outputs carry one rounding (2^-9 relative), fp32 only accumulation.
STEP_TOL = {"bf16": 1e-2, "f32": 1e-4}


@pytest.fixture(scope="module")
def ctx():
    import weight_mlp_layers_swiglu_b300 as pkg

    c = pkg.Context(0)
    yield c
    c.close()


@pytest.mark.parametrize("dt", ["bf16", "f32"])
@pytest.mark.parametrize("rows,d,f", [(300, 256, 384), (128, 64, 128), (1, 136, 264), (1000, 512, 1024)])
def test_swiglu_step(ctx, dt, rows, d, f):
    H = seeded((rows, d), 1.0, DT[dt], 1)
    Wg = seeded((f, d), d ** -0.5, DT[dt], 2)
    Wu = seeded((f, d), d ** -0.5, DT[dt], 3)
    Z = ctx.swiglu(H.cuda(), Wg.cuda(), Wu.cuda())
    assert ctx.sync() == 0
    ref = oracle.swiglu(H, Wg, Wu)
    assert rel_err(Z, ref) <= STEP_TOL[dt]


@pytest.mark.parametrize("dt", ["bf16", "f32"])
@pytest.mark.parametrize("B,T,d,k", [(2, 200, 320, 4), (1, 300, 256, 1), (3, 77, 128, 8), (1, 5, 72, 3)])
def test_target_step(ctx, dt, B, T, d, k):
    X0 = seeded((B, T, d), 0.02, DT[dt], 4)
    cw = seeded((d, k), k ** -0.5, DT[dt], 5)
    Wt = seeded((d, d), d ** -0.5, DT[dt], 6)
    scale = 1.0 / 128
    V, Y = ctx.target(X0.cuda(), cw.cuda(), Wt.cuda(), scale)
    assert ctx.sync() == 0
    for b in range(B):
        Y_ref = oracle.causal_conv(X0[b], cw)
        assert rel_err(Y[b], Y_ref) <= STEP_TOL[dt]
        assert rel_err(V[b], scale * oracle.target(X0[b], cw, Wt)) <= STEP_TOL[dt]


@pytest.mark.parametrize("dt", ["bf16", "f32"])
@pytest.mark.parametrize("B,T,d,f,C,w0", [
    (2, 300, 192, 384, 128, 1.0),    # ragged last chunk, ragged d and d_ff tiles
    (1, 1024, 256, 512, 256, 0.01),  # the fast part dominates: checks the prefix sums closely
    (3, 128, 128, 256, 128, 1.0),    # a single chunk per sequence
    (1, 5, 64, 64, 128, 1.0),        # fewer tokens than one tile
])
def test_chunk_state_step(ctx, dt, B, T, d, f, C, w0):
    V = seeded((B, T, d), 1.0, DT[dt], 7)
    Z = seeded((B, T, f), C ** -0.5, DT[dt], 8)
    W0 = seeded((d, f), w0, DT[dt], 9)
    W_eff, W_fin = ctx.chunk_state(V.cuda(), Z.cuda(), W0.cuda(), C)
    assert ctx.sync() == 0
    for b in range(B):
        ref_eff, ref_fin = oracle.chunk_weights(V[b], Z[b], W0, C, 1.0)
        assert rel_err(W_fin[b], ref_fin) <= (1e-3 if dt == "bf16" else 1e-5)
        assert rel_err(W_eff[b], ref_eff) <= STEP_TOL[dt]
        # the increments alone (what a broken scan would get wrong)
        fast = W_eff[b].double().cpu().numpy() - oracle._f64(W0)[None]
        ref_fast = ref_eff - oracle._f64(W0)[None]
        if np.abs(ref_fast).max() > 0:
            assert rel_err(fast, ref_fast) <= (5e-2 if dt == "bf16" else 1e-4)


@pytest.mark.parametrize("dt", ["bf16", "f32"])
@pytest.mark.parametrize("B,T,d,f,C", [(2, 300, 320, 384, 128), (1, 512, 256, 1024, 256), (1, 7, 64, 128, 128)])
def test_chunk_apply_step(ctx, dt, B, T, d, f, C):
    n = (T + C - 1) // C
    Z = seeded((B, T, f), 1.0, DT[dt], 10)
    W_eff = seeded((B, n, d, f), f ** -0.5, DT[dt], 11)
    O = ctx.chunk_apply(Z.cuda(), W_eff.cuda(), C)
    assert ctx.sync() == 0
    for b in range(B):
        assert rel_err(O[b], oracle.chunk_apply(Z[b], W_eff[b], C)) <= STEP_TOL[dt]


@pytest.mark.parametrize("fused", [True, False])
def test_steps_compose_to_the_layer(ctx, fused):
    """The layer call (fused state + apply kernel or two kernels) equals its documented step
    sequence, bit for bit."""
    import weight_mlp_layers_swiglu_b300 as pkg
    from weight_mlp_layers_swiglu_b300.inputs import random_case

    w, x = random_case(2, 384, 256, 512, 128, 4, 1.0 / 128, "bf16", 21)
    xd = {k: v.cuda() for k, v in x.items()}
    ctx.set_fused_tail(fused)
    O, Wf = ctx.layer_forward(xd["H"], xd["X0"], xd["W_gate"], xd["W_up"], xd["W_down0"], xd["W_target"],
                              xd["conv_w"], w.C, w.eta)
    ctx.set_fused_tail(True)
    Z = ctx.swiglu(xd["H"].view(-1, w.d), xd["W_gate"], xd["W_up"]).view(w.B, w.T, w.d_ff)
    V, _ = ctx.target(xd["X0"], xd["conv_w"], xd["W_target"], w.eta)
    W_eff, Wf2 = ctx.chunk_state(V, Z, xd["W_down0"], w.C)
    O2 = ctx.chunk_apply(Z, W_eff, w.C)
    assert ctx.sync() == 0
    assert torch.equal(O, O2) and torch.equal(Wf, Wf2)
    assert pkg.layer_launches(w.B, w.T, pkg.BF16) == 4
