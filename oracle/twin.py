"""Loader for the plain-C twin of the oracle (TEST INFRASTRUCTURE ONLY).

``build_twin()`` compiles oracle/twin.c with gcc into oracle/libipttt_twin.so;
``twin_layer_forward`` runs it on float64 copies of the inputs, one sequence at
a time.  Only the tests use it, on tiny inputs.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "twin.c")
_LIB = os.path.join(_HERE, "libipttt_twin.so")


def build_twin(force: bool = False) -> str:
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-O2", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"], check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    lib = ctypes.CDLL(build_twin())
    fn = lib.twin_sequence_forward
    dp = ctypes.POINTER(ctypes.c_double)
    fn.argtypes = [dp] * 7 + [ctypes.c_long] * 5 + [ctypes.c_double, dp, dp]
    fn.restype = ctypes.c_int
    return fn


def _f64c(x) -> np.ndarray:
    if hasattr(x, "detach"):
        import torch

        x = x.detach().to(torch.float64).cpu().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def twin_layer_forward(H, X0, W_gate, W_up, W_down0, W_target, conv_w, C: int, eta: float):
    fn = _load()
    H, X0 = _f64c(H), _f64c(X0)
    if H.ndim == 2:
        H, X0 = H[None], X0[None]
    Wg, Wu, W0, Wt, cw = (_f64c(a) for a in (W_gate, W_up, W_down0, W_target, conv_w))
    B, T, d = H.shape
    f = Wg.shape[0]
    k = cw.shape[1]
    O = np.zeros((B, T, d))
    Wf = np.zeros((B, d, f))
    ptr = lambda a: a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))
    for b in range(B):
        Hb, Xb = np.ascontiguousarray(H[b]), np.ascontiguousarray(X0[b])
        Ob = np.zeros((T, d))
        Wb = np.zeros((d, f))
        rc = fn(ptr(Hb), ptr(Xb), ptr(Wg), ptr(Wu), ptr(W0), ptr(Wt), ptr(cw),
                T, d, f, C, k, float(eta), ptr(Ob), ptr(Wb))
        if rc != 0:
            raise RuntimeError(f"twin_sequence_forward failed with code {rc}")
        O[b], Wf[b] = Ob, Wb
    return O, Wf
