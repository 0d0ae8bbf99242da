"""Context parallelism: one sequence split over ranks by token ranges.

This is the three-step scheme of the zhichai.net page ("In-Place TTT：给LLM装上"临时记忆插槽"，
让它边读边学", §3.2): Step 1, every rank computes the update total of its own chunks in parallel;
Step 2, one exclusive prefix sum over ranks gives each rank the fast weight at its first
token; Step 3, every rank applies its chunks from that weight in parallel.

Rank r holds a contiguous token range of every sequence.  Every range that has a non-empty
range after it must be a positive multiple of C (so that the ranks' chunks are the chunks of
the whole sequence) and hold at least k-1 tokens (so that the next rank's conv halo lies in
it); empty ranges may only come last.  cp_forward checks this on every rank before any data
moves.

The exchange is point to point along the ranks, and this module only moves buffers:
  * the halo: rank r sends its last k-1 X0 rows to rank r+1;
  * Step 2 as a chain: rank 0's starting state is W_down0; rank r receives its starting
    state P_r from rank r-1, forms P_{r+1} = P_r + S_r in place of its total S_r, and sends it
    to rank r+1.  The state travels in pieces, so that rank r+1 already receives the first
    pieces while rank r still adds the later ones.  Each rank holds one extra [B, d, d_ff]
    fp32 buffer (its P_r) whatever the number of ranks.
The arithmetic is injected: local_total (Step 1), prefix_step (the additions of Step 2) and
local_resume (Step 3) come from the library on a GPU (library_locals), or from any other
implementation of the same three calls, so the exchange logic itself runs on CPU ranks too.
"""
from __future__ import annotations

from typing import Callable, Optional

import torch

# local_total(H_r, X0_r, halo) -> S_r [B, d, d_ff] fp32: eta * sum over the rank's chunks of V_i^T Z_i
LocalTotal = Callable[[torch.Tensor, torch.Tensor, torch.Tensor], torch.Tensor]
# local_resume(H_r, X0_r, W_init, halo) -> (O_r [B, T_r, d], W_final_r [B, d, d_ff] fp32)
LocalResume = Callable[[torch.Tensor, torch.Tensor, torch.Tensor, torch.Tensor], tuple]
# prefix_step(P_in, W_down0, S, P_out, first, count): on the flattened elements
# [first, first + count) of the [B, d, d_ff] state, P_out = (P_in, or W_down0 broadcast over B
# when P_in is None) + (S, or zero when S is None); P_out may be P_in or S itself
PrefixStep = Callable[[Optional[torch.Tensor], torch.Tensor, Optional[torch.Tensor], torch.Tensor, int, int], None]

PIECES = 8  # pieces the state travels in along the chain


def check_ranges(lengths: list[int], C: int, k: int) -> None:
    """Raise ValueError unless the ranks' token ranges tile the sequence into whole chunks."""
    last = max((r for r, n in enumerate(lengths) if n > 0), default=-1)
    for r, n in enumerate(lengths):
        if n < 0:
            raise ValueError(f"rank {r} holds a negative number of tokens ({n})")
        if r < last:
            if n == 0:
                raise ValueError(f"rank {r} holds no tokens but rank {last} after it does: empty ranges come last")
            if n % C:
                raise ValueError(f"rank {r} holds {n} tokens, not a multiple of the chunk size C={C}")
            if n < k - 1:
                raise ValueError(f"rank {r} holds {n} tokens, fewer than the k-1={k - 1} the next rank's conv needs")


def halo_rows(X0_r: torch.Tensor, k: int) -> torch.Tensor:
    """The last k-1 X0 rows of a rank's range, [B, k-1, d] (what the next rank's conv needs)."""
    B, T_r, d = X0_r.shape
    out = torch.zeros((B, k - 1, d), dtype=X0_r.dtype, device=X0_r.device)
    n = min(k - 1, T_r)
    if n > 0:
        out[:, k - 1 - n:] = X0_r[:, T_r - n:]
    return out


def pieces(n: int, parts: int = PIECES) -> list[tuple[int, int]]:
    """[lo, hi) ranges that cut n elements into about `parts` pieces, each a multiple of 4 long
    (16-byte aligned fp32) except possibly the last."""
    per = -(-n // max(parts, 1))
    step = max(4, (per + 3) // 4 * 4)
    return [(lo, min(lo + step, n)) for lo in range(0, n, step)]


def cp_forward(H_r, X0_r, W_down0, k: int, C: int, local_total: LocalTotal, local_resume: LocalResume,
               prefix_step: PrefixStep, group=None, parts: int = PIECES):
    """The three steps on this rank of `group` (torch.distributed; None = the default group).

    Returns this rank's O_r and the state after its last chunk (on the last rank that holds
    tokens, the final fast weight of the whole sequence)."""
    import torch.distributed as dist

    world = dist.get_world_size(group)
    rank = dist.get_rank(group)
    mine = torch.tensor([H_r.shape[1]], dtype=torch.int64, device=H_r.device)
    lengths = [torch.zeros_like(mine) for _ in range(world)]
    dist.all_gather(lengths, mine, group=group)
    check_ranges([int(t.item()) for t in lengths], C, k)
    peer = lambda r: dist.get_global_rank(group, r) if group is not None else r  # noqa: E731
    # the conv halo from the previous rank
    halo = torch.zeros_like(halo_rows(X0_r, k))
    if k > 1:
        mine_halo = halo_rows(X0_r, k)
        reqs = [dist.isend(mine_halo, peer(rank + 1), group=group)] if rank + 1 < world else []
        if rank > 0:
            dist.recv(halo, peer(rank - 1), group=group)
        for q in reqs:
            q.wait()
    S_r = local_total(H_r, X0_r, halo)                                       # Step 1
    # Step 2: the chain, piece by piece
    W_init = torch.empty_like(S_r)
    if rank == 0:
        prefix_step(None, W_down0, None, W_init, 0, W_init.numel())          # P_0 = W_down0
    flat_in, flat_out = W_init.view(-1), S_r.view(-1)
    sends = []
    for lo, hi in pieces(W_init.numel(), parts):
        if rank > 0:
            dist.recv(flat_in[lo:hi], peer(rank - 1), group=group)           # P_r, this piece
        if rank + 1 < world:
            prefix_step(W_init, W_down0, S_r, S_r, lo, hi - lo)              # P_{r+1} = P_r + S_r
            sends.append(dist.isend(flat_out[lo:hi], peer(rank + 1), group=group))
    for q in sends:
        q.wait()
    return local_resume(H_r, X0_r, W_init, halo)                             # Step 3


def cp_forward_emulated(H, X0, W_down0, k: int, C: int, world: int, T_r: int, local_total: LocalTotal,
                        local_resume: LocalResume, prefix_step: PrefixStep):
    """All ranks of the scheme one after another in this process (no collective): rank r gets
    tokens [r*T_r, (r+1)*T_r).  The chain of Step 2 runs in rank order.  Returns the
    concatenated O and the final state."""
    ranges = [(min(r * T_r, H.shape[1]), min((r + 1) * T_r, H.shape[1])) for r in range(world)]
    check_ranges([hi - lo for lo, hi in ranges], C, k)
    halos = [torch.zeros_like(halo_rows(X0[:, :0], k))]
    for lo, hi in ranges[:-1]:
        halos.append(halo_rows(X0[:, lo:hi], k))
    totals = [local_total(H[:, lo:hi].contiguous(), X0[:, lo:hi].contiguous(), halos[r])
              for r, (lo, hi) in enumerate(ranges)]
    P = torch.empty_like(totals[0])
    prefix_step(None, W_down0, None, P, 0, P.numel())
    outs, W_last = [], None
    for r, (lo, hi) in enumerate(ranges):
        W_init = P.clone()
        if r + 1 < world:
            prefix_step(P, W_down0, totals[r], P, 0, P.numel())
        O_r, W_last = local_resume(H[:, lo:hi].contiguous(), X0[:, lo:hi].contiguous(), W_init, halos[r])
        outs.append(O_r)
    return torch.cat(outs, dim=1), W_last


def library_locals(ctx, W_gate, W_up, W_target, conv_w, C: int, eta: float):
    """local_total / local_resume / prefix_step backed by the CUDA library (a Context on this
    rank's GPU).

    local_total is Step 1 (ipttt_layer_totals): the range's update total from a zero state, with
    the range's Z and V kept; prefix_step is one hop of Step 2 (ipttt_prefix_step);
    local_resume is Step 3 (ipttt_layer_apply_saved) from the kept Z and V, so Z and V are
    computed once per range.  The Step 3 calls take the kept ranges in the order of the Step 1
    calls (one range per rank; the ranks emulated one after another in one process run all
    their Step 1 calls first, in rank order)."""
    from collections import deque

    saved = deque()

    def local_total(H_r, X0_r, halo):
        S, buf = ctx.layer_totals(H_r, X0_r, W_gate, W_up, W_target, conv_w, halo, C, eta)
        saved.append((H_r.shape[1], buf))
        return S

    def local_resume(H_r, X0_r, W_init, halo):
        T_r, buf = saved.popleft()
        if T_r != H_r.shape[1]:
            raise ValueError("Step 3 range does not match the Step 1 range kept first")
        return ctx.layer_apply_saved(W_init.contiguous(), T_r, C, buf, H_r.dtype)

    def prefix_step(P_in, W_down0, S, P_out, first, count):
        ctx.prefix_step(P_in, W_down0, S, P_out, first, count)

    return local_total, local_resume, prefix_step
