"""Shared helpers for the tests (no arithmetic of the layer lives here)."""
import numpy as np
import torch


def rel_err(x, ref) -> float:
    """max|x - ref| / max|ref| (the parity metric), computed in float64."""
    x = x.detach().double().cpu().numpy() if isinstance(x, torch.Tensor) else np.asarray(x, dtype=np.float64)
    ref = ref.detach().double().cpu().numpy() if isinstance(ref, torch.Tensor) else np.asarray(ref, dtype=np.float64)
    den = float(np.abs(ref).max()) if ref.size else 0.0
    num = float(np.abs(x - ref).max()) if ref.size else 0.0
    return num / den if den > 0 else num


def seeded(shape, std, dtype, seed, device="cpu"):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(*shape, generator=g) * std).to(dtype).to(device)


def to_dev(inputs: dict, device="cuda"):
    return {k: v.to(device).contiguous() for k, v in inputs.items()}


TOL = {"f32": 1e-4, "bf16": 2e-2}


FAST_TOL = {"f32": 1e-3, "bf16": 5e-2}


def _bf16(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(torch.bfloat16).double().numpy()


def layer_check(w, x, O, Wf, tol=None, fast_tol=None):
    """The bar on O and W_final against the oracle, then the fast parts.

    The oracle's reference is built from its own pinned pieces, per sequence: Z and V once,
    the per-chunk weights W_eff (sequential exclusive prefix) and the per-chunk apply.

    bf16 stores Z, every chunk weight W_eff[i] (whose bulk is W_down0) and O in bf16, so O
    carries roundings of 2^-9 |W_eff| and 2^-9 |O| that can be a sizeable fraction of a small
    fast part.  The fast-part check therefore measures O against the oracle's own Z and W_eff
    rounded to bf16, applied, and rounded to bf16 again (the storage precision of the bf16
    path), relative to the size of the fast part, after allowing one bf16 ulp of the largest
    output (fp32 and fp64 sums can round to neighbouring bf16 values): what remains is
    accumulation error, which a wrong prefix (inclusive, shifted, a dropped chunk) exceeds by
    far.  The plain ratio against the unrounded oracle, storage roundings included, is reported
    beside it as O_fast_plain (not bounded).  The fast part must be well above one bf16 ulp of O
    for the check to mean anything (small tests use eta of a few 1/C).  Returns the errors;
    raises AssertionError past a bound."""
    from oracle import oracle

    tol = tol or TOL[w.dtype]
    fast_tol = fast_tol or FAST_TOL[w.dtype]
    W0 = oracle._f64(x["W_down0"])
    errs = {"O": 0.0, "W_final": 0.0, "O_fast": 0.0, "W_fast": 0.0, "O_fast_plain": 0.0}
    o_num = o_den = w_num = w_den = 0.0
    for b in range(w.B):
        Z = oracle.swiglu(x["H"][b], x["W_gate"], x["W_up"])
        V = oracle.target(x["X0"][b], x["conv_w"], x["W_target"])
        W_eff, W_ref = oracle.chunk_weights(V, Z, W0, w.C, w.eta)
        O_ref = oracle.chunk_apply(Z, W_eff, w.C)
        O_b = O[b].detach().double().cpu().numpy() if isinstance(O, torch.Tensor) else np.asarray(O[b])
        Wf_b = Wf[b].detach().double().cpu().numpy() if isinstance(Wf, torch.Tensor) else np.asarray(Wf[b])
        o_num, o_den = max(o_num, float(np.abs(O_b - O_ref).max())), max(o_den, float(np.abs(O_ref).max()))
        w_num, w_den = max(w_num, float(np.abs(Wf_b - W_ref).max())), max(w_den, float(np.abs(W_ref).max()))
        if w.eta != 0 and w.T > w.C:
            fast = O_ref - Z @ W0.T
            if w.dtype == "bf16":
                O_q = _bf16(oracle.chunk_apply(_bf16(Z), _bf16(W_eff), w.C))
                # fp32 (GPU) and fp64 (here) sums may round to neighbouring bf16 values: allow
                # one bf16 ulp of the largest output, then measure the rest against the fast part
                ulp = 2.0 ** (np.floor(np.log2(np.abs(O_ref).max())) - 7)
                e = float(max(0.0, np.abs(O_b - O_q).max() - ulp) / np.abs(fast).max())
                # reported, not bounded: the plain ratio against the unrounded oracle, which also
                # carries the bf16 storage of every chunk weight and of O
                errs["O_fast_plain"] = max(errs["O_fast_plain"], rel_err(O_b - (O_ref - fast), fast))
            else:
                e = rel_err(O_b - (O_ref - fast), fast)
            errs["O_fast"] = max(errs["O_fast"], e)
        if w.eta != 0:
            errs["W_fast"] = max(errs["W_fast"], rel_err(Wf_b - W0, W_ref - W0))
        del Z, V, W_eff, O_ref
    errs["O"] = o_num / o_den if o_den > 0 else o_num
    errs["W_final"] = w_num / w_den if w_den > 0 else w_num
    assert errs["O"] <= tol, f"O err {errs}"
    assert errs["W_final"] <= tol, f"W_final err {errs}"
    assert errs["O_fast"] <= fast_tol, f"fast part of O, err {errs}"
    assert errs["W_fast"] <= fast_tol, f"fast part of W_final, err {errs}"
    return errs
