"""Step (2) as one kernel (the causal conv formed inside the W_target GEMM, Y never stored)
against the two-kernel path (the conv kernel, then the GEMM): the same bits for every output.

The fused kernel forms each bf16 Y value with the conv kernel's fp32 fma chain and feeds the
GEMM the same operands in the same order, so the layer's O and final state, the resumed
calls' outputs and the context-parallel totals must be bit-identical with the switch on and
off, across ragged token counts (tiles that end inside a sequence), several sequences, every
conv size k = 1..8, the shifted (next-token) window, a conv halo from an earlier call, and
widths that are not multiples of the 64-channel k-block or the 256-column tile."""
import pytest
import torch

from tests.util import TOL, rel_err, seeded, to_dev
from weight_mlp_layers_swiglu_b300.inputs import random_case

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ctx():
    import weight_mlp_layers_swiglu_b300 as pkg

    c = pkg.Context(0)
    yield c
    c.close()


def _layer(ctx, xd, w, fused, shift=0):
    ctx.set_fused_target(fused)
    ctx.set_target_shift(shift)
    try:
        O, Wf = ctx.layer_forward(xd["H"], xd["X0"], xd["W_gate"], xd["W_up"], xd["W_down0"], xd["W_target"],
                                  xd["conv_w"], w.C, w.eta)
        assert ctx.sync() == 0, ctx.last_error()
    finally:
        ctx.set_fused_target(False)
        ctx.set_target_shift(0)
    return O, Wf


CASES = [  # B, T, d, d_ff, C, k, shift
    (1, 512, 256, 512, 256, 4, 0),
    (2, 300, 256, 512, 128, 4, 0),     # tiles ending inside each sequence
    (3, 129, 128, 256, 128, 3, 1),     # one token past a 128-row block; shifted window
    (1, 1000, 200, 256, 128, 8, 0),    # d = 200: a partial k-block and column tile; k = 8
    (2, 640, 320, 384, 128, 1, 0),
    (1, 384, 512, 256, 128, 2, 1),
    (1, 256, 136, 128, 128, 5, 0),
    (2, 257, 264, 256, 256, 6, 1),
    (1, 700, 128, 128, 128, 7, 0),
    (1, 1, 128, 128, 128, 4, 1),       # one token
]


@pytest.mark.parametrize("B,T,d,f,C,k,shift", CASES)
def test_fused_target_layer_is_bit_identical(ctx, B, T, d, f, C, k, shift):
    w, x = random_case(B, T, d, f, C, k, 4.0 / C, "bf16", 500 + T + k)
    xd = to_dev(x)
    O1, W1 = _layer(ctx, xd, w, True, shift)
    O0, W0 = _layer(ctx, xd, w, False, shift)
    assert torch.equal(O1, O0) and torch.equal(W1, W0)
    # and within the bar of the oracle
    from oracle import oracle

    O_ref, W_ref = oracle.layer_forward(x["H"], x["X0"], x["W_gate"], x["W_up"], x["W_down0"], x["W_target"],
                                        x["conv_w"], w.C, w.eta, shift=shift)
    assert rel_err(O1, O_ref) <= TOL["bf16"] and rel_err(W1, W_ref) <= TOL["bf16"]


@pytest.mark.parametrize("k", [2, 4, 8])
def test_fused_target_with_a_conv_halo(ctx, k):
    """A resumed call: the X0 rows before the call's first token come from the halo."""
    B, T, d, f, C = 2, 384, 256, 256, 128
    w, x = random_case(B, T, d, f, C, k, 4.0 / C, "bf16", 600 + k)
    xd = to_dev(x)
    halo = seeded((B, k - 1, d), 0.02, torch.bfloat16, 601 + k, "cuda")
    W_state = (seeded((B, d, f), f ** -0.5, torch.float32, 602) + x["W_down0"].float()).cuda()
    outs = []
    for fused in (True, False):
        ctx.set_fused_target(fused)
        try:
            O, Ws, Ho = ctx.layer_resume(xd["H"], xd["X0"], xd["W_gate"], xd["W_up"], xd["W_target"], xd["conv_w"],
                                         W_state, halo, C, w.eta)
            assert ctx.sync() == 0, ctx.last_error()
        finally:
            ctx.set_fused_target(False)
        outs.append((O.clone(), Ws.clone(), Ho.clone()))
    assert all(torch.equal(a, b) for a, b in zip(*outs))


def test_fused_target_in_layer_totals(ctx):
    B, T, d, f, C, k = 2, 512, 256, 256, 128, 4
    w, x = random_case(B, T, d, f, C, k, 2.0 / C, "bf16", 700)
    xd = to_dev(x)
    halo = seeded((B, k - 1, d), 0.02, torch.bfloat16, 701, "cuda")
    res = []
    for fused in (True, False):
        ctx.set_fused_target(fused)
        try:
            S, _ = ctx.layer_totals(xd["H"], xd["X0"], xd["W_gate"], xd["W_up"], xd["W_target"], xd["conv_w"], halo,
                                    C, w.eta)
            assert ctx.sync() == 0, ctx.last_error()
        finally:
            ctx.set_fused_target(False)
        res.append(S.clone())
    assert torch.equal(res[0], res[1])
