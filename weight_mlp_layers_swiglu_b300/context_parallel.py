"""Context parallelism: one sequence split over ranks by token ranges.

This is the three-step scheme of the zhichai.net page ("In-Place TTT：给LLM装上"临时记忆插槽"，
让它边读边学", §3.2): Step 1, every rank computes the update total of its own chunks in parallel;
Step 2, one exclusive prefix sum over ranks gives each rank the fast weight at its first
token; Step 3, every rank applies its chunks from that weight in parallel.  Here Step 3 is
the resumable layer (ipttt_layer_forward_resume), which also takes the k-1 X0 rows before
the rank's first token (the causal conv's halo) from the previous rank.

Rank r holds tokens [r*T_r, (r+1)*T_r) of every sequence; T_r must be a multiple of C on
every rank but the last, so that the ranks' chunks are the chunks of the whole sequence.
The exchange is two all_gathers on the process group: the fp32 totals S_q [B, d, d_ff] and
the k-1 halo rows.  The per-rank compute is passed in (the library on a GPU, or any other
implementation of the same two calls), so the exchange logic itself runs on CPU ranks too.
"""
from __future__ import annotations

from typing import Callable

import torch

# local_total(H_r, X0_r, halo) -> S_r [B, d, d_ff] fp32: eta * sum over the rank's chunks of V_i^T Z_i
LocalTotal = Callable[[torch.Tensor, torch.Tensor, torch.Tensor], torch.Tensor]
# local_resume(H_r, X0_r, W_init, halo) -> (O_r [B, T_r, d], W_final_r [B, d, d_ff] fp32)
LocalResume = Callable[[torch.Tensor, torch.Tensor, torch.Tensor, torch.Tensor], tuple]


def halo_rows(X0_r: torch.Tensor, k: int) -> torch.Tensor:
    """The last k-1 X0 rows of a rank's range, [B, k-1, d] (what the next rank's conv needs)."""
    B, T_r, d = X0_r.shape
    out = torch.zeros((B, k - 1, d), dtype=X0_r.dtype, device=X0_r.device)
    n = min(k - 1, T_r)
    if n > 0:
        out[:, k - 1 - n:] = X0_r[:, T_r - n:]
    return out


def exclusive_prefix(W_down0: torch.Tensor, totals: list[torch.Tensor], rank: int) -> torch.Tensor:
    """Step 2 for one rank: W_down0 + sum of the totals of the ranks before it, [B, d, d_ff], in
    the totals' precision (fp32 from the library)."""
    B = totals[0].shape[0]
    acc = W_down0.to(totals[0].dtype).unsqueeze(0).expand(B, *W_down0.shape).clone()
    for q in range(rank):
        acc += totals[q].to(acc.device)
    return acc


def previous_halo(halos: list[torch.Tensor], rank: int) -> torch.Tensor:
    """The halo of rank `rank`: the previous rank's last k-1 rows (zeros for rank 0)."""
    return torch.zeros_like(halos[0]) if rank == 0 else halos[rank - 1]


def cp_forward(H_r, X0_r, W_down0, k: int, local_total: LocalTotal, local_resume: LocalResume,
               group=None):
    """The three steps on this rank of `group` (torch.distributed; None = the default group).

    Returns this rank's O_r and the state after its last chunk (on the last rank, the final
    fast weight of the whole sequence)."""
    import torch.distributed as dist

    world = dist.get_world_size(group)
    rank = dist.get_rank(group)
    if world == 1:  # nothing to exchange
        W_init = W_down0.float().unsqueeze(0).expand(H_r.shape[0], *W_down0.shape).contiguous()
        return local_resume(H_r, X0_r, W_init, torch.zeros_like(halo_rows(X0_r, k)))
    my_halo = halo_rows(X0_r, k)
    halos = [torch.empty_like(my_halo) for _ in range(world)]
    dist.all_gather(halos, my_halo.contiguous(), group=group)
    halo = previous_halo(halos, rank)
    S_r = local_total(H_r, X0_r, halo)                                   # Step 1
    totals = [torch.empty_like(S_r) for _ in range(world)]
    dist.all_gather(totals, S_r.contiguous(), group=group)               # the one exchange
    W_init = exclusive_prefix(W_down0, totals, rank)                      # Step 2
    return local_resume(H_r, X0_r, W_init.to(S_r.device), halo)          # Step 3


def cp_forward_emulated(H, X0, W_down0, k: int, world: int, T_r: int, local_total: LocalTotal,
                        local_resume: LocalResume):
    """All ranks of the scheme one after another in this process (no collective): rank r gets
    tokens [r*T_r, (r+1)*T_r).  Returns the concatenated O and the final state."""
    ranges = [(r * T_r, min((r + 1) * T_r, H.shape[1])) for r in range(world)]
    halos = [halo_rows(X0[:, lo:hi], k) for lo, hi in ranges]
    totals = []
    for r, (lo, hi) in enumerate(ranges):
        totals.append(local_total(H[:, lo:hi].contiguous(), X0[:, lo:hi].contiguous(), previous_halo(halos, r)))
    outs, W_last = [], None
    for r, (lo, hi) in enumerate(ranges):
        W_init = exclusive_prefix(W_down0, totals, r).to(totals[r].device)
        O_r, W_last = local_resume(H[:, lo:hi].contiguous(), X0[:, lo:hi].contiguous(), W_init,
                                   previous_halo(halos, r))
        outs.append(O_r)
    return torch.cat(outs, dim=1), W_last


def library_locals(ctx, W_gate, W_up, W_target, conv_w, C: int, eta: float):
    """local_total / local_resume backed by the CUDA library (a Context on this rank's GPU).

    local_total is Step 1 (ipttt_layer_totals): the range's update total from a zero state, with
    the range's Z and V kept; local_resume is Step 3 (ipttt_layer_apply_saved) from those, so Z
    and V are computed once per range.  The Step 3 calls take the kept ranges in the order of
    the Step 1 calls (one range per rank; the ranks emulated one after another in one process
    run all their Step 1 calls first, in rank order)."""
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

    return local_total, local_resume
