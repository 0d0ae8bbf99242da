"""Layer parity on the GPU: ipttt_layer_forward through the C ABI against the CPU oracle on the
same seeded inputs, with the bounds of the layer's specification: max|X - X_ref| / max|X_ref|
<= 1e-4 (fp32) and <= 2e-2 (bf16) for O and for the final W_down.  The fast parts alone
(O - Z W_down0^T and W_final - W_down0) are checked too, since W_down0 dominates both."""
import numpy as np
import pytest
import torch

from oracle import oracle
from tests.util import layer_check, to_dev
from weight_mlp_layers_swiglu_b300.inputs import WORKLOADS, make_inputs, random_case

pytestmark = pytest.mark.gpu

@pytest.fixture(scope="module")
def ctx():
    import weight_mlp_layers_swiglu_b300 as pkg

    c = pkg.Context(0)
    yield c
    c.close()


def run(ctx, w, x):
    xd = to_dev(x)
    O, Wf = ctx.layer_forward(xd["H"], xd["X0"], xd["W_gate"], xd["W_up"], xd["W_down0"], xd["W_target"],
                              xd["conv_w"], w.C, w.eta)
    assert ctx.sync() == 0, ctx.last_error()
    return O, Wf


def check(w, x, O, Wf):
    return layer_check(w, x, O, Wf)


def test_tiny_fp32_workload(ctx):
    """The fp32 workload at its full size: T=2048, d=256, d_ff=1024, C=256, k=4, eta=0.01."""
    w = WORKLOADS["tiny_fp32"]
    x = make_inputs(w)
    O, Wf = run(ctx, w, x)
    check(w, x, O, Wf)


@pytest.mark.parametrize("B,T,d,f,C,k,dt", [
    (1, 1024, 256, 512, 128, 4, "bf16"),    # 8 chunks
    (2, 1000, 256, 768, 128, 4, "bf16"),    # ragged last chunk, two sequences
    (1, 640, 320, 384, 256, 2, "bf16"),     # ragged d and d_ff tiles
    (3, 257, 128, 256, 128, 8, "bf16"),     # 3 sequences, 1-token last chunk
    (1, 777, 256, 512, 100, 4, "f32"),      # fp32, C not a multiple of anything
    (2, 300, 64, 128, 64, 1, "f32"),
])
def test_layer_small(ctx, B, T, d, f, C, k, dt):
    w, x = random_case(B, T, d, f, C, k, 4.0 / C, dt, 100 + T)
    O, Wf = run(ctx, w, x)
    check(w, x, O, Wf)


@pytest.mark.parametrize("dt", ["bf16", "f32"])
def test_single_token_and_single_chunk(ctx, dt):
    for T, C in ((1, 128), (128, 128), (100, 256)):
        w, x = random_case(1, T, 128, 256, C, 4, 0.5, dt, 7 + T)
        O, Wf = run(ctx, w, x)
        check(w, x, O, Wf)


@pytest.mark.parametrize("dt", ["bf16", "f32"])
def test_eta_zero_is_the_plain_mlp(ctx, dt):
    w, x = random_case(1, 512, 128, 256, 128, 4, 0.0, dt, 31)
    O, Wf = run(ctx, w, x)
    check(w, x, O, Wf)
    assert torch.equal(Wf[0].cpu(), x["W_down0"].float())


@pytest.mark.parametrize("dt", ["bf16", "f32"])
def test_empty_inputs(ctx, dt):
    w, x = random_case(2, 0, 64, 128, 128, 4, 0.1, dt, 3)
    O, Wf = run(ctx, w, x)
    assert O.shape == (2, 0, 64)
    for b in range(2):
        assert torch.equal(Wf[b].cpu(), x["W_down0"].float())
    w, x = random_case(0, 16, 64, 128, 128, 4, 0.1, dt, 3)
    O, Wf = run(ctx, w, x)
    assert O.numel() == 0 and Wf.numel() == 0


def test_causality_on_gpu(ctx):
    """Perturbing X0 inside chunk i leaves the GPU's O of chunks <= i bit-identical."""
    w, x = random_case(1, 1024, 256, 512, 128, 4, 1.0 / 128, "bf16", 44)
    O, _ = run(ctx, w, x)
    x2 = dict(x)
    x2["X0"] = x["X0"].clone()
    x2["X0"][0, 3 * 128 + 5] += 0.5
    O2, _ = run(ctx, w, x2)
    assert torch.equal(O[0, :4 * 128], O2[0, :4 * 128])
    assert not torch.equal(O[0, 4 * 128:], O2[0, 4 * 128:])


def test_deterministic(ctx):
    w, x = random_case(2, 512, 256, 512, 128, 4, 1.0 / 128, "bf16", 5)
    O1, W1 = run(ctx, w, x)
    O2, W2 = run(ctx, w, x)
    assert torch.equal(O1, O2) and torch.equal(W1, W2)


@pytest.mark.parametrize("dt,B,T,d,f,C,k", [
    ("bf16", 2, 384, 256, 512, 128, 4),     # one piece
    ("bf16", 2, 9000, 256, 512, 1024, 4),   # three pieces (4096, 4096, 808): uploads, compute and downloads overlap
    ("bf16", 1, 12288, 128, 256, 512, 1),   # 4096, 4096, then the last 4096 as 2048, 1024, 512, 512; no conv halo
    ("f32", 2, 5000, 64, 128, 48, 3),       # 4128, then 480, 240, 96, 48 and a ragged 8
])
def test_host_buffer_entry_point_matches(ctx, dt, B, T, d, f, C, k):
    """The host-buffer entry runs a call in pieces (multiples of C) whose copies overlap the
    compute; each piece resumes from the previous one's state and halo, so the result is the
    device entry's bit for bit."""
    w, x = random_case(B, T, d, f, C, k, 1.0 / C, dt, 6)
    O, Wf = run(ctx, w, x)
    xd = to_dev(x)
    H_h, X_h = x["H"].pin_memory(), x["X0"].pin_memory()
    O_h = torch.empty_like(x["H"]).pin_memory()
    W_h = torch.empty((w.B, w.d, w.d_ff), dtype=torch.float32).pin_memory()
    ctx.layer_forward_host(H_h, X_h, xd["W_gate"], xd["W_up"], xd["W_down0"], xd["W_target"], xd["conv_w"], w.C,
                           w.eta, O_h, W_h)
    assert ctx.sync() == 0
    assert torch.equal(O_h, O.cpu()) and torch.equal(W_h, Wf.cpu())


def test_argument_errors_launch_nothing(ctx):
    import weight_mlp_layers_swiglu_b300 as pkg

    w, x = random_case(1, 256, 128, 256, 128, 4, 0.1, "bf16", 8)
    xd = to_dev(x)
    O = torch.full((1, 256, 128), 7.0, dtype=torch.bfloat16, device="cuda")
    Wf = torch.full((1, 128, 256), 7.0, device="cuda")
    small_ws = torch.empty(1024, dtype=torch.uint8, device="cuda")
    with pytest.raises(pkg.IptttError) as e:
        ctx.layer_forward(xd["H"], xd["X0"], xd["W_gate"], xd["W_up"], xd["W_down0"], xd["W_target"], xd["conv_w"],
                          w.C, w.eta, O=O, W_final=Wf, workspace=small_ws)
    assert e.value.status == 3
    with pytest.raises(pkg.IptttError) as e:  # C not a multiple of 128 on the bf16 path
        ctx.layer_forward(xd["H"], xd["X0"], xd["W_gate"], xd["W_up"], xd["W_down0"], xd["W_target"], xd["conv_w"],
                          100, w.eta, O=O, W_final=Wf)
    assert e.value.status == 2
    with pytest.raises(pkg.IptttError) as e:  # output aliasing an input
        ctx.layer_forward(xd["H"], xd["X0"], xd["W_gate"], xd["W_up"], xd["W_down0"], xd["W_target"], xd["conv_w"],
                          w.C, w.eta, O=xd["H"].view(1, 256, 128), W_final=Wf)
    assert e.value.status == 1
    with pytest.raises(pkg.IptttError) as e:  # misaligned pointer
        Hm = torch.empty(1 * 256 * 128 + 1, dtype=torch.bfloat16, device="cuda")[1:].view(1, 256, 128)
        ctx.layer_forward(Hm, xd["X0"], xd["W_gate"], xd["W_up"], xd["W_down0"], xd["W_target"], xd["conv_w"],
                          w.C, w.eta, O=O, W_final=Wf)
    assert e.value.status == 1
    assert ctx.sync() == 0
    assert torch.all(O == 7.0) and torch.all(Wf == 7.0)


def test_device_wait_limit_reports_timeout_and_context_survives(ctx):
    ctx.set_wait_limit_ns(20_000_000)  # 20 ms
    ctx.selftest_wait_timeout()
    assert ctx.sync() == 5
    assert "gave up" in ctx.last_error()
    ctx.set_wait_limit_ns(2_000_000_000)
    w, x = random_case(1, 256, 128, 256, 128, 4, 4.0 / 128, "bf16", 9)
    O, Wf = run(ctx, w, x)
    check(w, x, O, Wf)


def test_timing_counts_launches(ctx):
    import weight_mlp_layers_swiglu_b300 as pkg

    w, x = random_case(1, 512, 256, 512, 128, 4, 1.0 / 128, "bf16", 10)
    xd = to_dev(x)

    def timed(fused_target):
        ctx.set_fused_target(fused_target)
        try:
            ctx.timing_begin()
            for _ in range(3):
                ctx.layer_forward(xd["H"], xd["X0"], xd["W_gate"], xd["W_up"], xd["W_down0"], xd["W_target"],
                                  xd["conv_w"], w.C, w.eta)
            return ctx.timing_read()
        finally:
            ctx.set_fused_target(False)

    # the conv as a kernel of its own, then the target GEMM (the default)
    ms, calls, launches = timed(False)
    assert calls == 3 and launches == 12  # SwiGLU, conv, target, fused state + apply
    assert launches == 3 * pkg.layer_launches(w.B, w.T, pkg.BF16)
    assert ms["apply"] == 0.0
    assert all(ms[s] > 0 for s in ("swiglu", "conv", "target", "state"))
    # step (2) as one kernel: the conv stage has zero length (event gaps only)
    ms, calls, launches = timed(True)
    assert calls == 3 and launches == 9
    assert all(ms[s] > 0 for s in ("swiglu", "target", "state")) and ms["conv"] < 3 * 0.01
