"""Context parallelism on the GPU, ranks emulated one after another on one device (no kernel
waits on another): the library computes each rank's total, the chain of prefix states and
each resumed range; the halo and the states are passed between them on the host side.  The
result must meet the parity bar against the oracle, and stay close to one call of the layer
(the per-rank totals sum the fp32 state in a different order, so a few bf16 roundings may
differ)."""
import pytest
import torch

from tests.util import TOL, rel_err, to_dev
from weight_mlp_layers_swiglu_b300.inputs import random_case

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dt,world,T_r", [("bf16", 2, 512), ("bf16", 4, 256), ("f32", 3, 192)])
def test_emulated_ranks_match_one_call(dt, world, T_r):
    import weight_mlp_layers_swiglu_b300 as pkg
    from weight_mlp_layers_swiglu_b300 import context_parallel as cp

    C = 128 if dt == "bf16" else 64
    w, x = random_case(2, world * T_r - 40, 256, 512, C, 4, 4.0 / C, dt, 91)
    xd = to_dev(x)
    ctx = pkg.Context(0)
    O_ref, W_ref = ctx.layer_forward(xd["H"], xd["X0"], xd["W_gate"], xd["W_up"], xd["W_down0"], xd["W_target"],
                                     xd["conv_w"], w.C, w.eta)
    lt, lr, ps = cp.library_locals(ctx, xd["W_gate"], xd["W_up"], xd["W_target"], xd["conv_w"], w.C, w.eta)
    O, W = cp.cp_forward_emulated(xd["H"], xd["X0"], xd["W_down0"], w.k, w.C, world, T_r, lt, lr, ps)
    assert ctx.sync() == 0, ctx.last_error()
    ctx.close()
    from oracle import oracle

    O_or, W_or = oracle.layer_forward(x["H"], x["X0"], x["W_gate"], x["W_up"], x["W_down0"], x["W_target"],
                                      x["conv_w"], w.C, w.eta)
    assert rel_err(O, O_or) <= TOL[dt] and rel_err(W, W_or) <= TOL[dt]
    assert rel_err(O, O_ref) <= TOL[dt] and rel_err(W, W_ref) <= TOL[dt] / 20


@pytest.mark.parametrize("dt,B,T,d,f,C,k", [("bf16", 2, 700, 256, 512, 256, 4), ("bf16", 1, 300, 192, 384, 128, 3),
                                          ("f32", 2, 200, 64, 128, 48, 4)])
def test_totals_and_apply_saved_match_resume(dt, B, T, d, f, C, k):
    """Step 1 (the update total from zero, Z and V kept) equals the final state of a resumed call
    from zero, and Step 3 from the kept Z and V equals the resumed call from the same state, bit
    for bit."""
    import weight_mlp_layers_swiglu_b300 as pkg
    from tests.util import seeded

    w, x = random_case(B, T, d, f, C, k, 2.0 / C, dt, 93)
    xd = to_dev(x)
    ctx = pkg.Context(0)
    halo = seeded((B, k - 1, d), 0.02, x["H"].dtype, 94, "cuda")
    zero = torch.zeros((B, d, f), dtype=torch.float32, device="cuda")
    _, S_ref, _ = ctx.layer_resume(xd["H"], xd["X0"], xd["W_gate"], xd["W_up"], xd["W_target"], xd["conv_w"], zero,
                                   halo, C, w.eta)
    S, saved = ctx.layer_totals(xd["H"], xd["X0"], xd["W_gate"], xd["W_up"], xd["W_target"], xd["conv_w"], halo, C,
                                w.eta)
    W_init = (seeded((B, d, f), f ** -0.5, torch.float32, 95) + x["W_down0"].float()).cuda()
    O_ref, W_ref, _ = ctx.layer_resume(xd["H"], xd["X0"], xd["W_gate"], xd["W_up"], xd["W_target"], xd["conv_w"],
                                       W_init, halo, C, w.eta)
    O, Wf = ctx.layer_apply_saved(W_init, T, C, saved, x["H"].dtype)
    assert ctx.sync() == 0, ctx.last_error()
    assert torch.equal(S, S_ref)
    assert torch.equal(O, O_ref) and torch.equal(Wf, W_ref)
    ctx.close()


@pytest.mark.parametrize("dt", [torch.bfloat16, torch.float32])
def test_prefix_step_is_one_fp32_addition_per_element(dt):
    """ipttt_prefix_step: rank 0's state is W_down0 widened to fp32 and broadcast over the batch;
    each later hop adds a total, elementwise and in place, over any range of the flattened
    state: the same bits as torch's fp32 addition, also when applied in pieces of odd lengths
    (the scalar path) and at offsets that are multiples of four (the vector path)."""
    import weight_mlp_layers_swiglu_b300 as pkg
    from tests.util import seeded

    B, d, f = 3, 64, 136
    ctx = pkg.Context(0)
    W0 = seeded((d, f), f ** -0.5, dt, 1, "cuda")
    S = seeded((B, d, f), 1e-2, torch.float32, 2, "cuda")
    P0 = torch.full((B, d, f), float("nan"), device="cuda")
    ctx.prefix_step(None, W0, None, P0)
    P1 = torch.full_like(P0, float("nan"))
    n = B * d * f
    for lo, hi in [(0, 1000), (1000, 1003), (1003, 5001), (5001, n)]:
        ctx.prefix_step(P0, W0, S, P1, lo, hi - lo)
    S2 = S.clone()
    ctx.prefix_step(P1, W0, S2, S2)  # in place into the total, as the chain forwards it
    assert ctx.sync() == 0, ctx.last_error()
    ref0 = W0.float()[None].expand(B, d, f)
    assert torch.equal(P0, ref0)
    assert torch.equal(P1, ref0 + S)
    assert torch.equal(S2, (ref0 + S) + S)
    # a range past the end launches nothing and reports INVALID_ARG
    with pytest.raises(pkg.IptttError):
        ctx.prefix_step(P0, W0, S, P1, n - 4, 8)
    ctx.close()
