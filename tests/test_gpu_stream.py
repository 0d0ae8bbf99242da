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


# The decode rows (CUDA cores) against the chunked call's tensor-core products: the same
# arithmetic in another summation order, each result rounded to the dtype once.
DECODE_VS_CHUNKED = {"bf16": 1e-2, "f32": 1e-5}


@pytest.mark.parametrize("exact", [True, False])
@pytest.mark.parametrize("dt,B,T,d,f,C,steps", [
    ("bf16", 2, 300, 128, 256, 128, [1] * 300),                    # token-by-token decoding
    ("bf16", 1, 700, 256, 512, 256, [1, 5, 250, 3, 2, 256, 100, 83]),  # mixed calls, CTA-pair chunks
    ("bf16", 2, 520, 128, 256, 128, [256, 1, 1, 1, 125, 136]),     # prefill, then decode
    ("bf16", 3, 400, 136, 264, 128, [8, 7, 1, 120, 8, 2, 254]),    # 8-token steps, widths off the tiles
    ("f32", 2, 200, 64, 128, 48, [7, 1, 40, 52, 100]),
])
def test_decode_with_chunk_buffer_matches_one_call(ctx, exact, dt, B, T, d, f, C, steps):
    """Calls of any length: tokens of an incomplete chunk are applied with the weight at the
    chunk's start and the chunk's update is committed when it completes.  After flush() the
    final state equals one call over the whole sequence bit for bit; so do the outputs with
    exact=True, and with the decode rows they agree to rounding and meet the oracle's bar."""
    import weight_mlp_layers_swiglu_b300 as pkg

    assert sum(steps) == T
    w, x = random_case(B, T, d, f, C, 4, 4.0 / C, dt, 90 + T)
    xd = to_dev(x)
    O_ref, W_ref = ctx.layer_forward(xd["H"], xd["X0"], xd["W_gate"], xd["W_up"], xd["W_down0"], xd["W_target"],
                                     xd["conv_w"], C, w.eta)
    O_ref, W_ref = O_ref.clone(), W_ref.clone()
    sl = pkg.StreamingLayer(ctx, xd["W_gate"], xd["W_up"], xd["W_down0"], xd["W_target"], xd["conv_w"], B, C, w.eta,
                            exact=exact)
    outs, lo = [], 0
    for n in steps:
        outs.append(sl.step(xd["H"][:, lo:lo + n].contiguous(), xd["X0"][:, lo:lo + n].contiguous()))
        lo += n
    sl.flush()
    assert ctx.sync() == 0, ctx.last_error()
    O = torch.cat(outs, dim=1)
    assert torch.equal(sl.state, W_ref)
    if exact:
        assert torch.equal(O, O_ref)
    else:
        assert rel_err(O, O_ref) <= DECODE_VS_CHUNKED[dt]
        O_or, _ = oracle.layer_forward(x["H"], x["X0"], x["W_gate"], x["W_up"], x["W_down0"], x["W_target"],
                                       x["conv_w"], C, w.eta)
        assert rel_err(O, O_or) <= TOL[dt]


@pytest.mark.parametrize("dt,B,m,d,f", [
    ("bf16", 1, 1, 2560, 9728),   # one token of the 4B-shaped layer
    ("bf16", 3, 2, 136, 264),
    ("bf16", 2, 8, 512, 1024),
    ("bf16", 5, 3, 64, 128),      # 15 SwiGLU rows: two launches of 8 and 7
    ("f32", 2, 5, 64, 136),
])
def test_decode_step_rows(ctx, dt, B, m, d, f):
    """ipttt_decode_step against the oracle's SwiGLU and chunk apply, against the tensor-core
    steps on the same rows, and its chunk-buffer stores (exact copies at tokens pos..)."""
    tdt = torch.bfloat16 if dt == "bf16" else torch.float32
    H = seeded((B, m, d), 1.0, tdt, 11 + m)
    X0 = seeded((B, m, d), 0.02, tdt, 12 + m)
    Wg = seeded((f, d), d ** -0.5, tdt, 13)
    Wu = seeded((f, d), d ** -0.5, tdt, 14)
    Wc = seeded((B, d, f), f ** -0.5, tdt, 15)
    C = 128  # the chunk buffer (and the chunk of the tensor-core apply)
    pos = C - m
    Hb = seeded((B, C, d), 3.0, tdt, 16, "cuda")
    Xb = seeded((B, C, d), 3.0, tdt, 17, "cuda")
    Hb0, Xb0 = Hb.clone(), Xb.clone()
    Hd, X0d, Wgd, Wud, Wcd = (t.cuda() for t in (H, X0, Wg, Wu, Wc))
    O, Z = ctx.decode_step(Hd, Wgd, Wud, Wcd, X0d, Hb, Xb, pos)
    Zc = ctx.swiglu(Hd.view(B * m, d), Wgd, Wud).view(B, m, f)
    Oc = ctx.chunk_apply(Zc, Wcd.view(B, 1, d, f), C)
    assert ctx.sync() == 0, ctx.last_error()
    for b in range(B):
        Z_ref = oracle.swiglu(H[b], Wg, Wu)
        O_ref = oracle.chunk_apply(Z_ref, Wc[b][None], C)
        assert rel_err(Z[b], Z_ref) <= TOL[dt], b
        assert rel_err(O[b], O_ref) <= TOL[dt], b
    assert rel_err(Z, Zc) <= DECODE_VS_CHUNKED[dt] and rel_err(O, Oc) <= DECODE_VS_CHUNKED[dt]
    assert torch.equal(Hb[:, pos:], Hd) and torch.equal(Xb[:, pos:], X0d)
    assert torch.equal(Hb[:, :pos], Hb0[:, :pos]) and torch.equal(Xb[:, :pos], Xb0[:, :pos])
    O2, Z2 = ctx.decode_step(Hd, Wgd, Wud, Wcd)  # without buffers; the same result on every run
    assert ctx.sync() == 0
    assert torch.equal(O2, O) and torch.equal(Z2, Z)


def test_decode_step_rejects_bad_calls(ctx):
    import weight_mlp_layers_swiglu_b300 as pkg

    B, d, f = 1, 64, 128
    W = seeded((f, d), 0.1, torch.bfloat16, 1, "cuda")
    Wc = seeded((B, d, f), 0.1, torch.bfloat16, 2, "cuda")
    H9 = seeded((B, 9, d), 1.0, torch.bfloat16, 3, "cuda")
    with pytest.raises(pkg.IptttError) as e:
        ctx.decode_step(H9, W, W, Wc)
    assert e.value.status == 2  # more than 8 tokens per sequence
    H = seeded((B, 4, d), 1.0, torch.bfloat16, 4, "cuda")
    buf = torch.zeros((B, 8, d), dtype=torch.bfloat16, device="cuda")
    buf2 = torch.zeros_like(buf)
    with pytest.raises(pkg.IptttError) as e:
        ctx.decode_step(H, W, W, Wc, H, buf, buf2, pos=5)  # tokens 5..8 past a buffer of 8
    assert e.value.status == 1
    with pytest.raises(pkg.IptttError) as e:
        ctx.decode_step(H, W, W, Wc, O=H)  # O overlaps H
    assert e.value.status == 1


def test_state_weight_rounds_the_state(ctx):
    W_state = seeded((2, 64, 128), 1.0, torch.float32, 91, "cuda")
    W = ctx.state_weight(W_state, torch.bfloat16)
    W32 = ctx.state_weight(W_state, torch.float32)
    assert ctx.sync() == 0
    assert torch.equal(W, W_state.to(torch.bfloat16)) and torch.equal(W32, W_state)


def test_decode_step_edge_cases(ctx):
    import weight_mlp_layers_swiglu_b300 as pkg

    d, f = 64, 128
    W = seeded((f, d), 0.1, torch.float32, 5, "cuda")
    # no sequences: nothing to do
    O, Z = ctx.decode_step(torch.empty((0, 1, d), device="cuda"), W, W, torch.empty((0, d, f), device="cuda"))
    assert ctx.sync() == 0 and O.shape == (0, 1, d) and Z.shape == (0, 1, f)
    # no tokens: unsupported (a step takes 1..8)
    with pytest.raises(pkg.IptttError) as e:
        ctx.decode_step(torch.empty((1, 0, d), device="cuda"), W, W, seeded((1, d, f), 0.1, torch.float32, 6, "cuda"))
    assert e.value.status == 2
    # fp32 with the chunk buffers: the stored rows are exact copies
    H = seeded((3, 2, d), 1.0, torch.float32, 7, "cuda")
    X0 = seeded((3, 2, d), 0.02, torch.float32, 8, "cuda")
    Hb = torch.zeros((3, 5, d), device="cuda")
    Xb = torch.zeros((3, 5, d), device="cuda")
    Wc = seeded((3, d, f), f ** -0.5, torch.float32, 9, "cuda")
    O, Z = ctx.decode_step(H, W, W, Wc, X0, Hb, Xb, pos=3)
    assert ctx.sync() == 0, ctx.last_error()
    assert torch.equal(Hb[:, 3:], H) and torch.equal(Xb[:, 3:], X0) and not Hb[:, :3].any() and not Xb[:, :3].any()
    for b in range(3):
        Z_ref = oracle.swiglu(H[b].cpu(), W.cpu(), W.cpu())
        assert rel_err(O[b], oracle.chunk_apply(Z_ref, Wc[b].cpu()[None], 2)) <= TOL["f32"]
