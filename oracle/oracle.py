"""CPU oracle for the In-Place TTT fast-weight SwiGLU layer.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import or run anything under ``oracle/``.
The product path (the CUDA library and its Python binding) never does, and it
shares no code, table or helper with this file.

A plain, slow, obviously correct restatement in float64 of what the layer
computes, written from these pages:

  [zhichai]    "In-Place TTT：给LLM装上"临时记忆插槽"，让它边读边学"
               (zhichai.net/topic/177981178) -- the only page with the
               layer's equations.
  [xiaoxiang]  "原位测试时训练" (xiaoxiang.io paper summary), section
               "核心方法", item 3 "高效的块状更新机制" -- the chunk ordering.
  [travelaiplan] the travelaiplan.net engineering blog, section 4 "分塊更新
               如何兼容長上下文與多請求並行" -- one fast-weight state per request.

Matrix products use numpy's matmul as a library step; nothing is blocked,
fused or reordered beyond the definitions below.  All inputs are widened
exactly to float64 first (bf16 and fp32 values are representable in fp64).

Readings taken where the pages are silent or garbled (also listed in the
design notes of the repository):
  * phi = SiLU ("SwiGLU"); no biases anywhere.
  * The loss printed as L = -<V, Z W_down>_F is shape-inconsistent; it is read
    as L = -<V, Z W_down^T>_F, whose negative gradient w.r.t. W_down is V^T Z,
    which is the printed update direction.
  * The causal Conv1D is depthwise (one k-tap filter per channel), zero
    left-padded by k-1 within each sequence, no bias; tap k-1 multiplies the
    current token, tap 0 the token k-1 steps back.
  * V = Conv1D(X0) W_target is taken literally: W_target is stored
    [d_in, d_out] and right-multiplies.
  * eta is applied as printed (no 1/C normalisation inside the layer).
  * Exactly one update per chunk; chunk i's output uses the weight left by
    chunks < i (exclusive prefix); the returned "final W_down" is the state
    after the last chunk's update.  The last chunk may be shorter than C.
  * A batch holds independent sequences: each has its own padding and its
    own fast-weight state; the frozen weights are shared.

Parity status: every function here is pinned by tests in tests/test_oracle_pins.py
and tests/test_oracle_stream.py
(hand-derived worked examples, closed forms, library routines, invariants and an
independent plain-C twin).  No function is "parity unpinned".
"""
from __future__ import annotations

import numpy as np


def _f64(x) -> np.ndarray:
    """Widen a numpy array or a CPU torch tensor (any float dtype) to float64."""
    if hasattr(x, "detach"):  # torch tensor, possibly bf16 (numpy has no bf16)
        import torch  # local: plain conversion only

        return x.detach().to(torch.float64).cpu().numpy()
    return np.asarray(x, dtype=np.float64)


def silu(a: np.ndarray) -> np.ndarray:
    """phi(a) = a * sigmoid(a) = a / (1 + exp(-a))  ([zhichai] §3.1, phi of the gated MLP)."""
    with np.errstate(over="ignore"):
        return a / (1.0 + np.exp(-a))


def swiglu(H, W_gate, W_up) -> np.ndarray:
    """Z = phi(H W_gate^T) ⊙ (H W_up^T)  ([zhichai] §3.1, gated-MLP equation).

    H: [T, d]; W_gate, W_up: [d_ff, d] (the equation's transposes); returns Z [T, d_ff].
    """
    H, W_gate, W_up = _f64(H), _f64(W_gate), _f64(W_up)
    return silu(H @ W_gate.T) * (H @ W_up.T)


def causal_conv(X0, conv_w, halo=None, shift: int = 0) -> np.ndarray:
    """Y = causal depthwise Conv1D(X0)  ([zhichai] §3.3, target equation, "causal padding").

    X0: [T, d]; conv_w: [d, k].  Y[t, c] = sum_s conv_w[c, s] * X0[t + shift - (k-1) + s, c].
    Token indices before 0 read `halo` ([k-1, d], the k-1 tokens that precede X0 when a
    sequence is processed in several calls) or are zero (left padding of k-1) without one.
    shift = 1 is the ablation variant whose window ends at the next token t+1 (the page
    describes the kernel size as setting how far ahead the target looks, and its Theorem 1
    uses the next token's embedding); the token after the last one reads as zero.
    """
    X0, conv_w = _f64(X0), _f64(conv_w)
    T, d = X0.shape
    k = conv_w.shape[1]
    pad = np.zeros((k - 1, d)) if halo is None else _f64(halo).reshape(k - 1, d)
    Xp = np.concatenate([pad, X0, np.zeros((shift, d))])  # Xp[t + k - 1] = X0[t]
    Y = np.zeros((T, d))
    for s in range(k):
        Y += conv_w[:, s] * Xp[s + shift: s + shift + T]
    return Y


def target(X0, conv_w, W_target, halo=None, shift: int = 0) -> np.ndarray:
    """V = Conv1D(X0) W_target  ([zhichai] §3.3, LM-aligned target).  Returns [T, d].

    W_target None is the "w/o Proj" ablation (identity projection, [zhichai] §6 table)."""
    Y = causal_conv(X0, conv_w, halo, shift)
    return Y if W_target is None else Y @ _f64(W_target)


def chunk_delta(V, Z) -> np.ndarray:
    """Delta W for one chunk: V_i^T Z_i  ([zhichai] §3.2 Step 1, §3.3 update rule).

    It is minus the gradient of L_i = -<V_i, Z_i W_down^T>_F with respect to W_down.
    V: [c, d], Z: [c, d_ff] for the c tokens of the chunk; returns [d, d_ff].
    """
    return _f64(V).T @ _f64(Z)


def chunk_rows(T: int, C: int):
    """Row ranges of the chunks: [iC, min((i+1)C, T)) for i = 0 .. ceil(T/C)-1  ([zhichai] §3.2)."""
    return [(s, min(s + C, T)) for s in range(0, T, C)]


def sequence_forward(H, X0, W_gate, W_up, W_down0, W_target, conv_w, C: int, eta: float, halo=None,
                     shift: int = 0):
    """One sequence, the literal sequential chunk loop.

    For each chunk in order: the chunk's output is computed with the current
    fast weight, then the fast weight takes one step
    W <- W + eta * V_i^T Z_i  ([zhichai] §3.2 bullets and §3.3 update rule;
    [xiaoxiang] "核心方法" item 3: output first with the previous weight, then update).
    W_down0 is the fast weight at the first token ([d, d_ff]); `halo` the k-1 X0 rows
    before it (see causal_conv).  Returns O [T, d] and the final W_down [d, d_ff].
    """
    Z = swiglu(H, W_gate, W_up)
    V = target(X0, conv_w, W_target, halo, shift)
    W = _f64(W_down0).copy()
    T = Z.shape[0]
    O = np.zeros((T, W.shape[0]))
    for lo, hi in chunk_rows(T, C):
        O[lo:hi] = Z[lo:hi] @ W.T
        W = W + eta * chunk_delta(V[lo:hi], Z[lo:hi])
    return O, W


def layer_forward(H, X0, W_gate, W_up, W_down0, W_target, conv_w, C: int, eta: float, shift: int = 0):
    """Batched layer: H, X0 [B, T, d] -> O [B, T, d], final W_down [B, d, d_ff].

    The sequences of a batch are independent; each carries its own fast-weight
    state and its own causal padding ([travelaiplan] §4, per-request state).
    """
    H, X0 = _f64(H), _f64(X0)
    if H.ndim == 2:
        H, X0 = H[None], X0[None]
    B, T, d = H.shape
    f = _f64(W_gate).shape[0]
    O = np.zeros((B, T, d))
    Wf = np.zeros((B, d, f))
    for b in range(B):
        O[b], Wf[b] = sequence_forward(H[b], X0[b], W_gate, W_up, W_down0, W_target, conv_w, C, eta,
                                       shift=shift)
    return O, Wf


def layer_resume(H, X0, W_gate, W_up, W_target, conv_w, W_state, X0_halo, C: int, eta: float):
    """Continue every sequence of a batch from where an earlier call left it.

    The fast weight is carried from call to call: the pages' stated direction is read-while-
    learn streaming inference with one fast-weight state per session ([zhichai] §9 future
    directions; [travelaiplan] §4).  W_state [B, d, d_ff] is each sequence's fast weight at its
    first token of this call; X0_halo [B, k-1, d] its k-1 preceding X0 rows (zeros at the start
    of a sequence).  Chunks are counted from this call's first token, so a sequence split at a
    multiple of C gives the same result as one call over the whole sequence.
    Returns O [B, T, d], the final state [B, d, d_ff] and the new halo [B, k-1, d] (the last
    k-1 rows of [X0_halo, X0]).
    """
    H, X0 = _f64(H), _f64(X0)
    W_state, X0_halo = _f64(W_state), _f64(X0_halo)
    B, T, d = H.shape
    k = _f64(conv_w).shape[1]
    f = _f64(W_gate).shape[0]
    O = np.zeros((B, T, d))
    Wf = np.zeros((B, d, f))
    halo_out = np.zeros((B, k - 1, d))
    for b in range(B):
        O[b], Wf[b] = sequence_forward(H[b], X0[b], W_gate, W_up, W_state[b], W_target, conv_w, C, eta,
                                       halo=X0_halo[b])
        halo_out[b] = np.concatenate([X0_halo[b], X0[b]])[T:]
    return O, Wf, halo_out


def chunk_weights(V, Z, W_down0, C: int, eta: float):
    """The weights each chunk is applied with, for one sequence.

    W_eff[i] = W_down0 + eta * sum_{j<i} V_j^T Z_j (the exclusive prefix of
    [zhichai] §3.2 Step 2), built by the same sequential update as
    sequence_forward.  Returns (W_eff [n, d, d_ff], final W_down [d, d_ff]).
    """
    V, Z = _f64(V), _f64(Z)
    W = _f64(W_down0).copy()
    out = []
    for lo, hi in chunk_rows(Z.shape[0], C):
        out.append(W.copy())
        W = W + eta * chunk_delta(V[lo:hi], Z[lo:hi])
    return np.stack(out) if out else np.zeros((0,) + W.shape), W


def chunk_apply(Z, W_eff, C: int) -> np.ndarray:
    """O_i = Z_i W_eff[i]^T for every chunk ([zhichai] §3.2 Step 3).  Z [T, d_ff] -> O [T, d]."""
    Z, W_eff = _f64(Z), _f64(W_eff)
    O = np.zeros((Z.shape[0], W_eff.shape[1]))
    for i, (lo, hi) in enumerate(chunk_rows(Z.shape[0], C)):
        O[lo:hi] = Z[lo:hi] @ W_eff[i].T
    return O
