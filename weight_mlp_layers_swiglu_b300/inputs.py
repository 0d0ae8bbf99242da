"""Seeded synthetic workloads for the fast-weight SwiGLU layer.

This module only draws random tensors of the right shapes and distributions.
It holds none of the layer's arithmetic, so the CPU oracle (under ``oracle/``)
and the CUDA path can both be fed from it without sharing any computation.

Workloads (shapes from the In-Place TTT pages: a Qwen3-4B-shaped MLP,
d=2560 / d_ff=9728, 32k and 128k contexts, chunk sizes 512-1024; the pages'
evaluation suites are not available, so these tensors stand in for them):

  name          B   T       d     d_ff  C     k  eta     dtype
  tiny_fp32     1   2048    256   1024  256   4  0.01    f32
  small_0p4b    1   32768   1024  4096  512   4  1/512   bf16
  qwen3_4b_32k  1   32768   2560  9728  1024  4  1/1024  bf16
  long_128k     1   131072  1024  4096  1024  4  1/1024  bf16
  serve_8x8k    8   8192    2560  9728  512   4  1/512   bf16

Distributions: H ~ N(0,1) (post-RMSNorm hidden state), X0 ~ N(0, 0.02^2)
(embedding output), W_gate, W_up, W_target ~ N(0, 1/d), W_down0 ~ N(0, 1/d_ff),
conv_w ~ N(0, 1/k).  Everything is drawn in fp32 from a torch CPU generator in
a fixed order -- W_gate, W_up, W_down0, W_target, conv_w with the workload
seed, then H_b and X0_b for each sequence b with seed + 1 + b -- and is then
rounded (round-to-nearest-even) to bf16 for the bf16 workloads.  The frozen
weights are shared by all sequences of a batch; every sequence has its own
H and X0.
"""
from __future__ import annotations

from dataclasses import dataclass, replace

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    T: int
    d: int
    d_ff: int
    C: int
    k: int
    eta: float
    dtype: str  # "f32" or "bf16"
    seed: int

    @property
    def n_chunks(self) -> int:
        return (self.T + self.C - 1) // self.C

    @property
    def tokens(self) -> int:
        return self.B * self.T

    def flops(self) -> float:
        """Algorithmic FLOPs of one layer call (state form).

        Per token: 4*d*d_ff for the two up-projections, 2*d*d_ff for the
        chunk update, 2*d*d_ff for the output projection, 2*d*d for the
        target projection and 2*k*d for the depthwise convolution.
        """
        per_tok = 8 * self.d * self.d_ff + 2 * self.d * self.d + 2 * self.k * self.d
        return float(self.B) * float(self.T) * float(per_tok)

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


WORKLOADS = {
    "tiny_fp32": Workload("tiny_fp32", 1, 2048, 256, 1024, 256, 4, 0.01, "f32", 0),
    "small_0p4b": Workload("small_0p4b", 1, 32768, 1024, 4096, 512, 4, 1.0 / 512, "bf16", 1),
    "qwen3_4b_32k": Workload("qwen3_4b_32k", 1, 32768, 2560, 9728, 1024, 4, 1.0 / 1024, "bf16", 2),
    "long_128k": Workload("long_128k", 1, 131072, 1024, 4096, 1024, 4, 1.0 / 1024, "bf16", 3),
    "serve_8x8k": Workload("serve_8x8k", 8, 8192, 2560, 9728, 512, 4, 1.0 / 512, "bf16", 4),
}

WORKLOAD_ORDER = ["tiny_fp32", "small_0p4b", "qwen3_4b_32k", "long_128k", "serve_8x8k"]


def _normal(gen: torch.Generator, shape, std: float) -> torch.Tensor:
    return torch.randn(*shape, generator=gen, dtype=torch.float32) * std


def torch_dtype(name: str) -> torch.dtype:
    if name == "f32":
        return torch.float32
    if name == "bf16":
        return torch.bfloat16
    raise ValueError(f"unknown dtype {name!r}")


def make_weights(w: Workload) -> dict:
    """Frozen weights, drawn with the workload seed, in the workload dtype (CPU)."""
    gen = torch.Generator().manual_seed(w.seed)
    d, f, k = w.d, w.d_ff, w.k
    out = {
        "W_gate": _normal(gen, (f, d), d ** -0.5),
        "W_up": _normal(gen, (f, d), d ** -0.5),
        "W_down0": _normal(gen, (d, f), f ** -0.5),
        "W_target": _normal(gen, (d, d), d ** -0.5),
        "conv_w": _normal(gen, (d, k), k ** -0.5),
    }
    dt = torch_dtype(w.dtype)
    return {n: t.to(dt) for n, t in out.items()}


def make_activations(w: Workload, b: int, T: int | None = None) -> tuple[torch.Tensor, torch.Tensor]:
    """H_b and X0_b for sequence b (seed + 1 + b), optionally only the first T tokens.

    Drawing the first T tokens gives exactly the leading rows of the full
    draw, so a prefix of a long workload can be regenerated cheaply.
    """
    T = w.T if T is None else T
    gen = torch.Generator().manual_seed(w.seed + 1 + b)
    H = _normal(gen, (w.T, w.d), 1.0)[:T]
    X0 = _normal(gen, (w.T, w.d), 0.02)[:T]
    dt = torch_dtype(w.dtype)
    return H.to(dt).contiguous(), X0.to(dt).contiguous()


def make_inputs(w: Workload, T: int | None = None) -> dict:
    """All inputs of one layer call as CPU tensors: weights plus H, X0 of shape [B, T, d]."""
    out = make_weights(w)
    Hs, Xs = [], []
    for b in range(w.B):
        H, X0 = make_activations(w, b, T)
        Hs.append(H)
        Xs.append(X0)
    T_eff = w.T if T is None else T
    dt = torch_dtype(w.dtype)
    out["H"] = torch.stack(Hs).contiguous() if Hs else torch.empty((0, T_eff, w.d), dtype=dt)
    out["X0"] = torch.stack(Xs).contiguous() if Xs else torch.empty((0, T_eff, w.d), dtype=dt)
    return out


def random_case(B: int, T: int, d: int, d_ff: int, C: int, k: int, eta: float, dtype: str,
                seed: int) -> tuple[Workload, dict]:
    """A small workload of arbitrary shape with the same distributions (for tests)."""
    w = Workload(f"case_{B}x{T}_{d}_{d_ff}_{C}_{k}", B, T, d, d_ff, C, k, eta, dtype, seed)
    return w, make_inputs(w)
