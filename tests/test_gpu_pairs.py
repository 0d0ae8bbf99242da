"""The bf16 GEMMs on CTA pairs (tcgen05.mma.cta_group::2, 256-row tiles) against the same GEMMs on
single CTAs (128-row tiles), through the C ABI: every output element is the same fp32 sum of the
same products in the same K order, so the two tilings must agree bit for bit.  The shapes end in
ragged tails (rows that fill only the even CTA of the last pair, ragged d and d_ff) and the
oracle bounds the pair path too (the step tests run it by default)."""
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
    c.set_cta_pairs(True)
    c.close()


def both(ctx, fn):
    ctx.set_cta_pairs(True)
    a = fn()
    assert ctx.sync() == 0, ctx.last_error()
    ctx.set_cta_pairs(False)
    b = fn()
    assert ctx.sync() == 0, ctx.last_error()
    ctx.set_cta_pairs(True)
    return a, b


@pytest.mark.parametrize("rows,d,f", [(300, 256, 384), (128, 64, 128), (1, 136, 264), (1000, 512, 1024),
                                      (257, 2560, 1024)])
def test_swiglu_pairs_match_single(ctx, rows, d, f):
    H = seeded((rows, d), 1.0, torch.bfloat16, 1, "cuda")
    Wg = seeded((f, d), d ** -0.5, torch.bfloat16, 2, "cuda")
    Wu = seeded((f, d), d ** -0.5, torch.bfloat16, 3, "cuda")
    a, b = both(ctx, lambda: ctx.swiglu(H, Wg, Wu).clone())
    assert torch.equal(a, b)
    assert rel_err(a, oracle.swiglu(H.cpu(), Wg.cpu(), Wu.cpu())) <= 1e-2


@pytest.mark.parametrize("B,T,d", [(2, 200, 320), (1, 300, 256), (3, 77, 128), (1, 600, 2560)])
def test_target_pairs_match_single(ctx, B, T, d):
    X0 = seeded((B, T, d), 0.02, torch.bfloat16, 4, "cuda")
    cw = seeded((d, 4), 0.5, torch.bfloat16, 5, "cuda")
    Wt = seeded((d, d), d ** -0.5, torch.bfloat16, 6, "cuda")
    a, b = both(ctx, lambda: ctx.target(X0, cw, Wt, 1.0 / 128)[0].clone())
    assert torch.equal(a, b)


@pytest.mark.parametrize("B,T,d,f,C", [(2, 600, 320, 384, 256), (1, 1024, 256, 1024, 512), (1, 100, 128, 256, 256),
                                       (2, 300, 192, 384, 128)])
def test_apply_pairs_match_single(ctx, B, T, d, f, C):
    n = (T + C - 1) // C
    Z = seeded((B, T, f), f ** -0.5, torch.bfloat16, 7, "cuda")
    W = seeded((B * n, d, f), 1.0, torch.bfloat16, 8, "cuda").view(B, n, d, f)
    a, b = both(ctx, lambda: ctx.chunk_apply(Z, W, C).clone())
    assert torch.equal(a, b)
    for bb in range(B):
        assert rel_err(a[bb], oracle.chunk_apply(Z[bb].cpu(), W[bb].cpu(), C)) <= 1e-2


# tail: "unfused" = the state and apply kernels; the fused kernel with its apply tiles chosen per
# call ("auto"), 256 x 256 ("narrow") or 256 x 512 ("wide")
@pytest.mark.parametrize("tail", ["unfused", "auto", "narrow", "wide"])
@pytest.mark.parametrize("B,T,d,f,C,k", [
    (2, 700, 256, 512, 256, 4),
    (1, 1100, 384, 768, 512, 3),
    (3, 600, 1024, 4096, 256, 4),   # 192 pair units: more unit pairs than co-resident CTA pairs
    (4, 9472, 512, 256, 256, 4),    # 148 apply tiles of 256 x 512, two waves of wide tiles
    (2, 9472, 640, 256, 256, 3),    # wide tiles whose second 256-column half lies past d
    (2, 700, 200, 328, 256, 4),     # widths that are not multiples of 64: V and Z through 3-D maps
])
def test_layer_pairs_match_single(ctx, tail, B, T, d, f, C, k):
    w, x = random_case(B, T, d, f, C, k, 2.0 / C, "bf16", 60 + T)
    xd = to_dev(x)
    ctx.set_fused_tail(tail != "unfused")
    ctx.set_apply_tiles({"unfused": 0, "auto": 0, "narrow": 1, "wide": 2}[tail])
    try:
        (Oa, Wa), (Ob, Wb) = both(ctx, lambda: tuple(t.clone() for t in ctx.layer_forward(
            xd["H"], xd["X0"], xd["W_gate"], xd["W_up"], xd["W_down0"], xd["W_target"], xd["conv_w"], C, w.eta)))
    finally:
        ctx.set_fused_tail(True)
        ctx.set_apply_tiles(0)
    assert torch.equal(Oa, Ob) and torch.equal(Wa, Wb)
    O_ref, W_ref = oracle.layer_forward(x["H"], x["X0"], x["W_gate"], x["W_up"], x["W_down0"], x["W_target"],
                                        x["conv_w"], C, w.eta)
    assert rel_err(Oa, O_ref) <= TOL["bf16"] and rel_err(Wa, W_ref) <= TOL["bf16"]


@pytest.mark.parametrize("reverse_case", [False, True])
@pytest.mark.parametrize("B,T,d,f,C", [(2, 300, 192, 384, 128), (1, 1024, 512, 1024, 256), (3, 130, 136, 264, 128),
                                       (1, 5, 64, 64, 128), (3, 600, 1024, 4096, 256)])
def test_chunk_state_pairs_match_single(ctx, reverse_case, B, T, d, f, C):
    """The state kernel on pairs (256-row units) and on single CTAs (128-row units); the reverse
    scan is exercised through the backward pass.  Widths that are multiples of 64 (192 x 384,
    512 x 1024, 64 x 64, 1024 x 4096) give the pairs V and Z as blocks of 64 columns (one 4-D TMA
    request per operand and k-block, d = 192 and d = 64 with the second block of a CTA past the
    edge); 136 x 264 keeps the 3-D maps; the single CTAs always load 3-D maps."""
    if not reverse_case:
        V = seeded((B, T, d), 1.0, torch.bfloat16, 7, "cuda")
        Z = seeded((B, T, f), C ** -0.5, torch.bfloat16, 8, "cuda")
        W0 = seeded((d, f), 1.0, torch.bfloat16, 9, "cuda")
        (Ea, Fa), (Eb, Fb) = both(ctx, lambda: tuple(t.clone() for t in ctx.chunk_state(V, Z, W0, C)))
        assert torch.equal(Ea, Eb) and torch.equal(Fa, Fb)
        for b in range(B):
            ref_eff, ref_fin = oracle.chunk_weights(V[b].cpu(), Z[b].cpu(), W0.cpu(), C, 1.0)
            assert rel_err(Fa[b], ref_fin) <= 1e-3 and rel_err(Ea[b], ref_eff) <= 1e-2
    else:
        w, x = random_case(B, T, d, f, C, 3, 2.0 / C, "bf16", 70 + T)
        xd = to_dev(x)
        dO = seeded((B, T, d), 1.0, torch.bfloat16, 71, "cuda")
        dWf = seeded((B, d, f), 0.5, torch.float32, 72, "cuda")
        ga, gb = both(ctx, lambda: {k: (None if v is None else v.clone()) for k, v in ctx.layer_backward(
            xd["H"], xd["X0"], xd["W_gate"], xd["W_up"], xd["W_down0"], xd["W_target"], xd["conv_w"], C, w.eta, dO,
            dWf).items()})
        for k in ga:
            assert torch.equal(ga[k], gb[k]), k


@pytest.mark.parametrize("B,T,d,f,C", [(2, 700, 256, 512, 256), (1, 600, 384, 768, 512)])
def test_resume_pairs_match_single(ctx, B, T, d, f, C):
    """The resumed layer (each sequence from its own fp32 state; the fused kernel then writes and
    publishes W_eff[b, 0] itself) on pairs and on single CTAs, and against the oracle."""
    w, x = random_case(B, T, d, f, C, 4, 2.0 / C, "bf16", 80 + T)
    xd = to_dev(x)
    W_state = (seeded((B, d, f), f ** -0.5, torch.float32, 81) + x["W_down0"].float()).cuda()
    halo = seeded((B, 3, d), 0.02, torch.bfloat16, 82, "cuda")
    (Oa, Wa, ha), (Ob, Wb, hb) = both(ctx, lambda: tuple(t.clone() for t in ctx.layer_resume(
        xd["H"], xd["X0"], xd["W_gate"], xd["W_up"], xd["W_target"], xd["conv_w"], W_state, halo, C, w.eta)))
    assert torch.equal(Oa, Ob) and torch.equal(Wa, Wb) and torch.equal(ha, hb)
    O_ref, W_ref, _ = oracle.layer_resume(x["H"], x["X0"], x["W_gate"], x["W_up"], x["W_target"], x["conv_w"],
                                          W_state.cpu(), halo.cpu(), C, w.eta)
    assert rel_err(Oa, O_ref) <= TOL["bf16"] and rel_err(Wa, W_ref) <= TOL["bf16"]


def test_apply_tile_width_argument(ctx):
    """ipttt_set_apply_tiles takes 0 (per call), 1 or 2 and refuses anything else."""
    import weight_mlp_layers_swiglu_b300 as pkg

    for h in (1, 2, 0):
        ctx.set_apply_tiles(h)
    for bad in (-1, 3):
        with pytest.raises(pkg.IptttError) as e:
            ctx.set_apply_tiles(bad)
        assert e.value.status == 1
