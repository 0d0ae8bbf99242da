"""Seeded random shapes through the C ABI against the oracle: the layer (both dtypes, every kernel
path the shape selects: CTA pairs or single CTAs, fused or not), the resumed layer and the
backward pass.  The shapes are drawn to land on tile edges and off them (d and d_ff multiples of
8, T around multiples of C and of the 128/256-row tiles, C a multiple of 128 for bf16)."""
import numpy as np
import pytest
import torch

from oracle import oracle
from oracle.oracle_grad import layer_backward
from tests.util import TOL, rel_err, seeded, to_dev
from weight_mlp_layers_swiglu_b300.inputs import random_case

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ctx():
    import weight_mlp_layers_swiglu_b300 as pkg

    c = pkg.Context(0)
    yield c
    c.set_cta_pairs(True)
    c.set_fused_tail(True)
    c.close()


def draw(seed: int):
    r = np.random.default_rng(seed)
    dt = "bf16" if r.random() < 0.75 else "f32"
    B = int(r.integers(1, 4))
    d = int(r.choice([64, 128, 136, 192, 256, 264, 384, 520]))
    f = int(r.choice([128, 264, 384, 512, 776, 1024]))
    C = int(r.choice([128, 256, 384, 512])) if dt == "bf16" else int(r.choice([16, 48, 64, 100, 128]))
    k = int(r.integers(1, 9))
    T = int(r.choice([1, C - 1, C, C + 1, 2 * C + 7, 3 * C, 255, 257, 700]))
    T = max(T, 1)
    pairs = bool(r.random() < 0.7)
    fused = bool(r.random() < 0.8)
    return dt, B, T, d, f, C, k, pairs, fused


@pytest.mark.parametrize("seed", range(24))
def test_random_shape_forward_and_backward(ctx, seed):
    dt, B, T, d, f, C, k, pairs, fused = draw(seed)
    w, x = random_case(B, T, d, f, C, k, 2.0 / C, dt, 4000 + seed)
    xd = to_dev(x)
    ctx.set_cta_pairs(pairs)
    ctx.set_fused_tail(fused)
    O, Wf = ctx.layer_forward(xd["H"], xd["X0"], xd["W_gate"], xd["W_up"], xd["W_down0"], xd["W_target"],
                              xd["conv_w"], C, w.eta)
    dO = seeded((B, T, d), 1.0, x["H"].dtype, 5000 + seed, "cuda")
    dWf = seeded((B, d, f), 0.5, torch.float32, 6000 + seed, "cuda")
    g = ctx.layer_backward(xd["H"], xd["X0"], xd["W_gate"], xd["W_up"], xd["W_down0"], xd["W_target"],
                           xd["conv_w"], C, w.eta, dO, dWf)
    assert ctx.sync() == 0, ctx.last_error()
    O_ref, W_ref = oracle.layer_forward(x["H"], x["X0"], x["W_gate"], x["W_up"], x["W_down0"], x["W_target"],
                                        x["conv_w"], C, w.eta)
    shape = (dt, B, T, d, f, C, k, pairs, fused)
    assert rel_err(O, O_ref) <= TOL[dt], shape
    assert rel_err(Wf, W_ref) <= TOL[dt], shape
    ref = layer_backward(x["H"], x["X0"], x["W_gate"], x["W_up"], x["W_down0"], x["W_target"], x["conv_w"], C, w.eta,
                         dO.cpu(), dWf.cpu())
    for n, v in ref.items():
        assert rel_err(g[n], v) <= TOL[dt], (n, shape)


@pytest.mark.parametrize("seed", range(8))
def test_random_shape_resume(ctx, seed):
    dt, B, T, d, f, C, k, pairs, fused = draw(100 + seed)
    w, x = random_case(B, T, d, f, C, k, 2.0 / C, dt, 7000 + seed)
    xd = to_dev(x)
    ctx.set_cta_pairs(pairs)
    ctx.set_fused_tail(fused)
    W_state = (seeded((B, d, f), f ** -0.5, torch.float32, 7100 + seed) + x["W_down0"].float()).cuda()
    halo = seeded((B, k - 1, d), 0.02, x["H"].dtype, 7200 + seed, "cuda")
    O, Ws, h = ctx.layer_resume(xd["H"], xd["X0"], xd["W_gate"], xd["W_up"], xd["W_target"], xd["conv_w"], W_state,
                                halo, C, w.eta)
    assert ctx.sync() == 0, ctx.last_error()
    O_ref, W_ref, h_ref = oracle.layer_resume(x["H"], x["X0"], x["W_gate"], x["W_up"], x["W_target"], x["conv_w"],
                                              W_state.cpu(), halo.cpu(), C, w.eta)
    shape = (dt, B, T, d, f, C, k, pairs, fused)
    assert rel_err(O, O_ref) <= TOL[dt], shape
    assert rel_err(Ws, W_ref) <= TOL[dt], shape
    assert torch.equal(h.cpu().double(), torch.from_numpy(h_ref)), shape


@pytest.mark.parametrize("seed", range(12))
def test_random_shape_decode_step(ctx, seed):
    """ipttt_decode_step on drawn shapes (1..8 tokens of 1..6 sequences, widths on and off the
    tiles, both dtypes) against the oracle's SwiGLU and chunk apply."""
    r = np.random.default_rng(9000 + seed)
    dt = "bf16" if r.random() < 0.7 else "f32"
    tdt = torch.bfloat16 if dt == "bf16" else torch.float32
    B = int(r.integers(1, 7))
    m = int(r.integers(1, 9))
    d = int(r.choice([8, 64, 136, 256, 520, 1032]))
    f = int(r.choice([8, 128, 264, 776, 2056]))
    H = seeded((B, m, d), 1.0, tdt, 9100 + seed)
    Wg = seeded((f, d), d ** -0.5, tdt, 9200 + seed)
    Wu = seeded((f, d), d ** -0.5, tdt, 9300 + seed)
    Wc = seeded((B, d, f), f ** -0.5, tdt, 9400 + seed)
    O, Z = ctx.decode_step(H.cuda(), Wg.cuda(), Wu.cuda(), Wc.cuda())
    assert ctx.sync() == 0, ctx.last_error()
    shape = (dt, B, m, d, f)
    for b in range(B):
        Z_ref = oracle.swiglu(H[b], Wg, Wu)
        assert rel_err(Z[b], Z_ref) <= TOL[dt], (b, shape)
        assert rel_err(O[b], oracle.chunk_apply(Z_ref, Wc[b][None], m)) <= TOL[dt], (b, shape)
