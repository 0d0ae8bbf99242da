"""Streaming / resumable layer on the GPU (ipttt_layer_forward_resume through the C ABI).

A resumed call continues every sequence from its fp32 fast-weight state and X0 conv halo.
It is checked against the oracle's resumable layer, and a sequence cut at multiples of C and
fed call by call must reproduce one call over the whole sequence bit for bit."""
import pytest
import torch

from oracle import oracle
from tests.util import TOL, rel_err, seeded, to_dev
from weight_mlp_layers_swiglu_b300.inputs import random_case

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ctx():
    import weight_mlp_layers_swiglu_b300 as pkg

    c = pkg.Context(0)
    yield c
    c.close()


@pytest.mark.parametrize("dt,B,T,d,f,C,k", [
    ("bf16", 2, 640, 256, 512, 128, 4),
    ("bf16", 1, 300, 192, 384, 128, 3),   # ragged last chunk and tiles
    ("f32", 2, 200, 64, 128, 48, 4),
    ("bf16", 1, 2, 128, 256, 128, 4),     # fewer tokens than the halo
])
def test_resume_matches_oracle(ctx, dt, B, T, d, f, C, k):
    w, x = random_case(B, T, d, f, C, k, 2.0 / C, dt, 500 + T)
    xd = to_dev(x)
    tdt = xd["H"].dtype
    W_state = (seeded((B, d, f), f ** -0.5, torch.float32, 7) + x["W_down0"].float()).cuda()
    halo = seeded((B, k - 1, d), 0.02, tdt, 8, "cuda")
    O, Ws, h = ctx.layer_resume(xd["H"], xd["X0"], xd["W_gate"], xd["W_up"], xd["W_target"], xd["conv_w"], W_state,
                                halo, C, w.eta)
    assert ctx.sync() == 0, ctx.last_error()
    O_ref, W_ref, h_ref = oracle.layer_resume(x["H"], x["X0"], x["W_gate"], x["W_up"], x["W_target"], x["conv_w"],
                                              W_state.cpu(), halo.cpu(), C, w.eta)
    assert rel_err(O, O_ref) <= TOL[dt]
    assert rel_err(Ws, W_ref) <= TOL[dt]
    assert torch.equal(h.cpu().double(), torch.from_numpy(h_ref))


@pytest.mark.parametrize("fused", [True, False])
@pytest.mark.parametrize("dt,cuts", [("bf16", [256, 768]), ("bf16", [128 * i for i in range(1, 8)]),
                                     ("f32", [64, 320])])
def test_stream_cut_at_chunk_multiples_is_bit_exact(ctx, fused, dt, cuts):
    import weight_mlp_layers_swiglu_b300 as pkg

    C = 128 if dt == "bf16" else 64
    w, x = random_case(2, 1000, 256, 512, C, 4, 4.0 / C, dt, 77)
    xd = to_dev(x)
    ctx.set_fused_tail(fused)
    try:
        O_ref, W_ref = ctx.layer_forward(xd["H"], xd["X0"], xd["W_gate"], xd["W_up"], xd["W_down0"],
                                         xd["W_target"], xd["conv_w"], C, w.eta)
        sl = pkg.StreamingLayer(ctx, xd["W_gate"], xd["W_up"], xd["W_down0"], xd["W_target"], xd["conv_w"], w.B, C,
                                w.eta)
        outs = []
        for lo, hi in zip([0] + cuts, cuts + [w.T]):
            outs.append(sl.step(xd["H"][:, lo:hi].contiguous(), xd["X0"][:, lo:hi].contiguous()))
        sl.flush()  # the sequence ends inside a chunk: commit that chunk's update
        assert ctx.sync() == 0, ctx.last_error()
    finally:
        ctx.set_fused_tail(True)
    assert torch.equal(torch.cat(outs, dim=1), O_ref)
    assert torch.equal(sl.state, W_ref)


def test_decode_steps_of_one_chunk(ctx):
    """Feeding C tokens per call (the decode path) gives the whole-sequence result."""
    import weight_mlp_layers_swiglu_b300 as pkg

    w, x = random_case(1, 1024, 256, 512, 128, 4, 4.0 / 128, "bf16", 78)
    xd = to_dev(x)
    O_ref, W_ref = ctx.layer_forward(xd["H"], xd["X0"], xd["W_gate"], xd["W_up"], xd["W_down0"], xd["W_target"],
                                     xd["conv_w"], w.C, w.eta)
    sl = pkg.StreamingLayer(ctx, xd["W_gate"], xd["W_up"], xd["W_down0"], xd["W_target"], xd["conv_w"], 1, 128, w.eta)
    outs = [sl.step(xd["H"][:, t:t + 128].contiguous(), xd["X0"][:, t:t + 128].contiguous()) for t in range(0, 1024, 128)]
    assert ctx.sync() == 0
    assert torch.equal(torch.cat(outs, dim=1), O_ref) and torch.equal(sl.state, W_ref)


def test_empty_resume_keeps_state_and_halo(ctx):
    w, x = random_case(2, 0, 64, 128, 128, 4, 0.1, "bf16", 3)
    xd = to_dev(x)
    W_state = seeded((2, 64, 128), 1.0, torch.float32, 9, "cuda")
    halo = seeded((2, 3, 64), 1.0, torch.bfloat16, 10, "cuda")
    O, Ws, h = ctx.layer_resume(xd["H"], xd["X0"], xd["W_gate"], xd["W_up"], xd["W_target"], xd["conv_w"], W_state,
                                halo, 128, 0.1)
    assert ctx.sync() == 0
    assert torch.equal(Ws, W_state) and torch.equal(h, halo)


def test_resume_rejects_overlapping_halo(ctx):
    import weight_mlp_layers_swiglu_b300 as pkg

    w, x = random_case(1, 256, 128, 256, 128, 4, 0.1, "bf16", 4)
    xd = to_dev(x)
    W_state = torch.zeros((1, 128, 256), device="cuda")
    halo = torch.zeros((1, 3, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(pkg.IptttError) as e:
        ctx.layer_resume(xd["H"], xd["X0"], xd["W_gate"], xd["W_up"], xd["W_target"], xd["conv_w"], W_state, halo,
                         128, 0.1, X0_halo_out=halo)
    assert e.value.status == 1


@pytest.mark.parametrize("dt,B,T,d,f,C,steps", [
    ("bf16", 2, 300, 128, 256, 128, [1] * 300),                    # token-by-token decoding
    ("bf16", 1, 700, 256, 512, 256, [1, 5, 250, 3, 2, 256, 100, 83]),  # mixed calls, CTA-pair chunks
    ("bf16", 2, 520, 128, 256, 128, [256, 1, 1, 1, 125, 136]),     # prefill, then decode
    ("f32", 2, 200, 64, 128, 48, [7, 1, 40, 52, 100]),
])
def test_decode_with_chunk_buffer_matches_one_call(ctx, dt, B, T, d, f, C, steps):
    """Calls of any length: tokens of an incomplete chunk are applied with the weight at the
    chunk's start and the chunk's update is committed when it completes; outputs, and after
    flush() the final state, equal one call over the whole sequence bit for bit."""
    import weight_mlp_layers_swiglu_b300 as pkg

    assert sum(steps) == T
    w, x = random_case(B, T, d, f, C, 4, 4.0 / C, dt, 90 + T)
    xd = to_dev(x)
    O_ref, W_ref = ctx.layer_forward(xd["H"], xd["X0"], xd["W_gate"], xd["W_up"], xd["W_down0"], xd["W_target"],
                                     xd["conv_w"], C, w.eta)
    O_ref, W_ref = O_ref.clone(), W_ref.clone()
    sl = pkg.StreamingLayer(ctx, xd["W_gate"], xd["W_up"], xd["W_down0"], xd["W_target"], xd["conv_w"], B, C, w.eta)
    outs, lo = [], 0
    for n in steps:
        outs.append(sl.step(xd["H"][:, lo:lo + n].contiguous(), xd["X0"][:, lo:lo + n].contiguous()))
        lo += n
    sl.flush()
    assert ctx.sync() == 0, ctx.last_error()
    assert torch.equal(torch.cat(outs, dim=1), O_ref)
    assert torch.equal(sl.state, W_ref)


def test_state_weight_rounds_the_state(ctx):
    W_state = seeded((2, 64, 128), 1.0, torch.float32, 91, "cuda")
    W = ctx.state_weight(W_state, torch.bfloat16)
    W32 = ctx.state_weight(W_state, torch.float32)
    assert ctx.sync() == 0
    assert torch.equal(W, W_state.to(torch.bfloat16)) and torch.equal(W32, W_state)
