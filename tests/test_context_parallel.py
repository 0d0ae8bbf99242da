"""Context parallelism (the zhichai.net page's §3.2 three-step scheme) on CPU ranks.

Each gloo rank holds a contiguous token range of every sequence and computes with the oracle;
the exchange (the k-1 halo rows to the next rank, and Step 2 as a rank-to-rank chain of the
prefix states, in pieces) runs through weight_mlp_layers_swiglu_b300.context_parallel.  The
concatenated outputs and the last rank's state must equal the oracle's single-process layer."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

from oracle import oracle
from weight_mlp_layers_swiglu_b300 import context_parallel as cp
from weight_mlp_layers_swiglu_b300.inputs import random_case

CASE = dict(B=2, T=48, d=6, f=10, C=8, k=3, eta=0.3, dtype="f32", seed=17)


def _oracle_locals(x, C, eta):
    def local_total(H_r, X0_r, halo):
        B, _, d = H_r.shape
        zero = np.zeros((B, d, x["W_gate"].shape[0]))
        _, S, _ = oracle.layer_resume(H_r, X0_r, x["W_gate"], x["W_up"], x["W_target"], x["conv_w"], zero, halo, C,
                                      eta)
        return torch.from_numpy(S)

    def local_resume(H_r, X0_r, W_init, halo):
        O, W, _ = oracle.layer_resume(H_r, X0_r, x["W_gate"], x["W_up"], x["W_target"], x["conv_w"], W_init, halo, C,
                                      eta)
        return torch.from_numpy(O), torch.from_numpy(W)

    return local_total, local_resume


def _prefix_step(P_in, W_down0, S, P_out, first, count):
    """Step 2's hop in float64 on CPU tensors (the test's stand-in for ipttt_prefix_step)."""
    n = P_out.numel()
    base = P_in.reshape(-1) if P_in is not None else W_down0.reshape(-1).to(P_out.dtype).repeat(n // W_down0.numel())
    out = base[first:first + count].clone()
    if S is not None:
        out += S.reshape(-1)[first:first + count]
    P_out.view(-1)[first:first + count] = out


def _inputs():
    w, x = random_case(CASE["B"], CASE["T"], CASE["d"], CASE["f"], CASE["C"], CASE["k"], CASE["eta"], CASE["dtype"],
                       CASE["seed"])
    return w, {n: t.double() for n, t in x.items()}


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, T_r, q, parts=8):
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w, x = _inputs()
    lo, hi = min(rank * T_r, w.T), min((rank + 1) * T_r, w.T)
    lt, lr = _oracle_locals(x, w.C, w.eta)
    try:
        O_r, W_r = cp.cp_forward(x["H"][:, lo:hi].contiguous(), x["X0"][:, lo:hi].contiguous(), x["W_down0"], w.k,
                                 w.C, lt, lr, _prefix_step, parts=parts)
        q.put((rank, O_r.numpy(), W_r.numpy()))
    except ValueError as e:
        q.put((rank, "ValueError", str(e)))
    dist.destroy_process_group()


def _spawn(world, T_r, parts=8):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, T_r, q, parts)) for r in range(world)]
    for p in procs:
        p.start()
    got = sorted([q.get(timeout=180) for _ in procs], key=lambda t: t[0])
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    return got


@pytest.mark.parametrize("world,T_r,parts", [(2, 24, 8), (3, 16, 8), (3, 24, 3), (4, 16, 8), (2, 40, 1),
                                             (1, 48, 8)])
def test_gloo_ranks_equal_the_single_process_layer(world, T_r, parts):
    got = _spawn(world, T_r, parts)
    w, x = _inputs()
    O_ref, W_ref = oracle.layer_forward(x["H"], x["X0"], x["W_gate"], x["W_up"], x["W_down0"], x["W_target"],
                                        x["conv_w"], w.C, w.eta)
    O = np.concatenate([g[1] for g in got if g[1].shape[1] > 0], axis=1)
    assert np.abs(O - O_ref).max() / np.abs(O_ref).max() < 1e-12
    # the last rank that holds tokens carries the final state of the whole sequence
    last = max(r for r in range(world) if r * T_r < w.T)
    assert np.abs(got[last][2] - W_ref).max() / np.abs(W_ref).max() < 1e-12


def test_ranges_that_do_not_tile_whole_chunks_are_refused_on_every_rank():
    """A non-final range that is not a multiple of C (here 20 tokens with C = 8), or an empty
    range before a non-empty one, is refused by every rank alike before any data moves."""
    for world, T_r in ((2, 20), (3, 4)):
        got = _spawn(world, T_r)
        assert all(g[1] == "ValueError" for g in got), got


def test_range_checks():
    cp.check_ranges([16, 16, 16], 8, 4)
    cp.check_ranges([16, 5, 0, 0], 8, 4)  # the last non-empty range may be ragged; empty ones trail
    for bad in ([12, 16], [16, 0, 8], [0, 8]):
        with pytest.raises(ValueError):
            cp.check_ranges(bad, 8, 4)
    with pytest.raises(ValueError):  # shorter than the next rank's conv halo (k - 1 = 4 rows)
        cp.check_ranges([2, 2], 2, 5)


def test_emulated_ranks_and_the_chain():
    w, x = _inputs()
    lt, lr = _oracle_locals(x, w.C, w.eta)
    O, W = cp.cp_forward_emulated(x["H"], x["X0"], x["W_down0"], w.k, w.C, 3, 16, lt, lr, _prefix_step)
    O_ref, W_ref = oracle.layer_forward(x["H"], x["X0"], x["W_gate"], x["W_up"], x["W_down0"], x["W_target"],
                                        x["conv_w"], w.C, w.eta)
    assert np.abs(O.numpy() - O_ref).max() / np.abs(O_ref).max() < 1e-12
    assert np.abs(W.numpy() - W_ref).max() / np.abs(W_ref).max() < 1e-12
    # the halo is the previous range's last k-1 rows
    X = torch.arange(2 * 5 * 3, dtype=torch.float64).reshape(2, 5, 3)
    assert torch.equal(cp.halo_rows(X, 3), X[:, 3:])
    # the pieces tile the state, each a multiple of 4 elements but the last
    for n in (1, 5, 64, 1001):
        p = cp.pieces(n, 8)
        assert p[0][0] == 0 and p[-1][1] == n and all(a[1] == b[0] for a, b in zip(p, p[1:]))
        assert all((hi - lo) % 4 == 0 for lo, hi in p[:-1])


def test_library_locals_keep_step_one_buffers_in_order():
    """The library glue on a stand-in context: Step 3 takes the Z and V that Step 1 kept, range
    by range in Step 1's order, and refuses a range whose length differs."""

    class FakeCtx:
        def __init__(self):
            self.calls = []

        def layer_totals(self, H_r, X0_r, W_gate, W_up, W_target, conv_w, halo, C, eta):
            buf = torch.full((4,), float(len(self.calls)))
            self.calls.append(("totals", H_r.shape[1]))
            return torch.zeros(H_r.shape[0], 2, 3), buf

        def layer_apply_saved(self, W_init, T, C, saved, dtype):
            self.calls.append(("apply", T, float(saved[0])))
            return torch.zeros(W_init.shape[0], T, 2, dtype=dtype), W_init

    fake = FakeCtx()
    lt, lr, _ = cp.library_locals(fake, None, None, None, None, 8, 0.1)
    H = [torch.zeros(2, n, 2) for n in (16, 8)]
    for h in H:
        lt(h, h, None)
    W = torch.zeros(2, 2, 3)
    lr(H[0], H[0], W, None)
    lr(H[1], H[1], W, None)
    assert fake.calls == [("totals", 16), ("totals", 8), ("apply", 16, 0.0), ("apply", 8, 1.0)]
    lt(H[0], H[0], None)
    with pytest.raises(ValueError):
        lr(H[1], H[1], W, None)
