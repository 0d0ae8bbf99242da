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
