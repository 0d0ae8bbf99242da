"""ctypes binding of libipttt.so (include/ipttt.h).

Argument marshalling only: torch tensors are checked for device, dtype, shape and
contiguity, and their data pointers are passed to the C ABI together with the
current CUDA stream.  Every step of the layer runs in the library's kernels; there
is no Python or CPU fallback -- if the library is missing, load() raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

IPTTT_OK = 0
STATUS_NAMES = {0: "OK", 1: "INVALID_ARG", 2: "UNSUPPORTED", 3: "WORKSPACE", 4: "CUDA", 5: "TIMEOUT"}
F32, BF16 = 0, 1
STAGES = ["swiglu", "conv", "target", "state", "apply"]

_lib = None

c_i64 = ctypes.c_int64
c_vp = ctypes.c_void_p

# name -> (restype, argtypes)
_SIGNATURES = {
    "ipttt_version": (ctypes.c_char_p, []),
    "ipttt_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "ipttt_create": (ctypes.c_int, [ctypes.POINTER(c_vp), ctypes.c_int, c_vp]),
    "ipttt_set_stream": (ctypes.c_int, [c_vp, c_vp]),
    "ipttt_set_wait_limit_ns": (ctypes.c_int, [c_vp, ctypes.c_uint64]),
    "ipttt_set_fused_tail": (ctypes.c_int, [c_vp, ctypes.c_int]),
    "ipttt_set_apply_tiles": (ctypes.c_int, [c_vp, ctypes.c_int]),
    "ipttt_set_fused_target": (ctypes.c_int, [c_vp, ctypes.c_int]),
    "ipttt_set_cta_pairs": (ctypes.c_int, [c_vp, ctypes.c_int]),
    "ipttt_set_target_shift": (ctypes.c_int, [c_vp, ctypes.c_int]),
    "ipttt_sync": (ctypes.c_int, [c_vp]),
    "ipttt_last_error": (ctypes.c_char_p, [c_vp]),
    "ipttt_destroy": (None, [c_vp]),
    "ipttt_workspace_size": (ctypes.c_int, [c_i64] * 5 + [ctypes.c_int, ctypes.c_int, ctypes.POINTER(ctypes.c_size_t)]),
    "ipttt_host_workspace_size": (ctypes.c_int,
                                  [c_i64] * 5 + [ctypes.c_int, ctypes.c_int, ctypes.POINTER(ctypes.c_size_t)]),
    "ipttt_layer_forward": (ctypes.c_int, [c_vp] * 8 + [c_i64] * 5 + [ctypes.c_int, ctypes.c_float, ctypes.c_int,
                                                                     c_vp, c_vp, c_vp, ctypes.c_size_t]),
    "ipttt_layer_forward_resume": (ctypes.c_int, [c_vp] * 9 + [c_i64] * 5 + [ctypes.c_int, ctypes.c_float,
                                                                            ctypes.c_int, c_vp, c_vp, c_vp, c_vp,
                                                                            ctypes.c_size_t]),
    "ipttt_layer_forward_host": (ctypes.c_int, [c_vp] * 8 + [c_i64] * 5 + [ctypes.c_int, ctypes.c_float,
                                                                          ctypes.c_int, c_vp, c_vp, c_vp,
                                                                          ctypes.c_size_t]),
    "ipttt_backward_workspace_size": (ctypes.c_int,
                                      [c_i64] * 5 + [ctypes.c_int, ctypes.c_int, ctypes.POINTER(ctypes.c_size_t)]),
    "ipttt_layer_backward": (ctypes.c_int, [c_vp] * 8 + [c_i64] * 5 + [ctypes.c_int, ctypes.c_float, ctypes.c_int]
                             + [c_vp] * 10 + [ctypes.c_size_t]),
    "ipttt_saved_size": (ctypes.c_int, [c_i64] * 5 + [ctypes.c_int, ctypes.c_int, ctypes.POINTER(ctypes.c_size_t)]),
    "ipttt_backward_saved_workspace_size": (ctypes.c_int, [c_i64] * 5 + [ctypes.c_int, ctypes.c_int,
                                                                         ctypes.POINTER(ctypes.c_size_t)]),
    "ipttt_layer_forward_train": (ctypes.c_int, [c_vp] * 8 + [c_i64] * 5 + [ctypes.c_int, ctypes.c_float, ctypes.c_int]
                                  + [c_vp] * 3 + [ctypes.c_size_t]),
    "ipttt_layer_backward_saved": (ctypes.c_int, [c_vp] * 7 + [c_i64] * 5 + [ctypes.c_int, ctypes.c_float, ctypes.c_int,
                                                                             c_vp, ctypes.c_size_t] + [c_vp] * 10
                                   + [ctypes.c_size_t]),
    "ipttt_state_weight": (ctypes.c_int, [c_vp, c_vp] + [c_i64] * 3 + [ctypes.c_int, c_vp]),
    "ipttt_decode_step": (ctypes.c_int, [c_vp] * 6 + [c_i64] * 4 + [ctypes.c_int] + [c_vp] * 4 + [c_i64] * 2),
    "ipttt_layer_totals": (ctypes.c_int, [c_vp] * 8 + [c_i64] * 5 + [ctypes.c_int, ctypes.c_float, ctypes.c_int,
                                                                     c_vp, c_vp, ctypes.c_size_t]),
    "ipttt_layer_apply_saved": (ctypes.c_int, [c_vp, c_vp] + [c_i64] * 5 + [ctypes.c_int, c_vp, ctypes.c_size_t, c_vp,
                                                                             c_vp]),
    "ipttt_prefix_step": (ctypes.c_int, [c_vp] * 4 + [c_i64] * 3 + [ctypes.c_int, c_i64, c_i64, c_vp]),
    "ipttt_swiglu": (ctypes.c_int, [c_vp] * 4 + [c_i64] * 3 + [ctypes.c_int, c_vp]),
    "ipttt_target": (ctypes.c_int, [c_vp] * 4 + [c_i64] * 3 + [ctypes.c_int, ctypes.c_float, ctypes.c_int, c_vp, c_vp]),
    "ipttt_chunk_state": (ctypes.c_int, [c_vp] * 4 + [c_i64] * 5 + [ctypes.c_int, c_vp, c_vp]),
    "ipttt_chunk_apply": (ctypes.c_int, [c_vp] * 3 + [c_i64] * 5 + [ctypes.c_int, c_vp]),
    "ipttt_target_noalloc": (ctypes.c_int, [c_vp] * 3 + [c_i64] * 3 + [ctypes.c_int, ctypes.c_float, ctypes.c_int,
                                                                    c_vp, c_vp, c_vp]),
    "ipttt_timing_begin": (ctypes.c_int, [c_vp]),
    "ipttt_timing_read": (ctypes.c_int, [c_vp, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(c_i64),
                                         ctypes.POINTER(c_i64)]),
    "ipttt_layer_launches": (c_i64, [c_i64, c_i64, ctypes.c_int]),
    "ipttt_selftest_wait_timeout": (ctypes.c_int, [c_vp]),
    "ipttt_sm_count": (ctypes.c_int, [c_vp]),
}


def exported_symbols() -> list[str]:
    return list(_SIGNATURES)


def load(build_if_missing: bool = True):
    """Load libipttt.so (building it first if it is missing or stale)."""
    global _lib
    if _lib is not None:
        return _lib
    if build_if_missing:
        _build.build()
    if not os.path.exists(_build.LIB_PATH):
        raise RuntimeError(f"CUDA library {_build.LIB_PATH} is missing; run weight_mlp_layers_swiglu_b300.build")
    lib = ctypes.CDLL(_build.LIB_PATH)
    for name, (res, args) in _SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


class IptttError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


def dtype_code(dt: torch.dtype) -> int:
    if dt == torch.bfloat16:
        return BF16
    if dt == torch.float32:
        return F32
    raise TypeError(f"unsupported dtype {dt}")


def workspace_size(B, T, d, d_ff, C, k, dtype: int, host: bool = False) -> int:
    lib = load()
    out = ctypes.c_size_t(0)
    fn = lib.ipttt_host_workspace_size if host else lib.ipttt_workspace_size
    st = fn(B, T, d, d_ff, C, k, dtype, ctypes.byref(out))
    if st != IPTTT_OK:
        raise IptttError(st, f"workspace_size(B={B}, T={T}, d={d}, d_ff={d_ff}, C={C}, k={k})")
    return out.value


def backward_workspace_size(B, T, d, d_ff, C, k, dtype: int) -> int:
    return _size_query("ipttt_backward_workspace_size", B, T, d, d_ff, C, k, dtype)


def _size_query(fn: str, B, T, d, d_ff, C, k, dtype: int) -> int:
    out = ctypes.c_size_t(0)
    st = getattr(load(), fn)(B, T, d, d_ff, C, k, dtype, ctypes.byref(out))
    if st != IPTTT_OK:
        raise IptttError(st, f"{fn}(B={B}, T={T}, d={d}, d_ff={d_ff}, C={C}, k={k})")
    return out.value


def saved_size(B, T, d, d_ff, C, k, dtype: int) -> int:
    return _size_query("ipttt_saved_size", B, T, d, d_ff, C, k, dtype)


def backward_saved_workspace_size(B, T, d, d_ff, C, k, dtype: int) -> int:
    return _size_query("ipttt_backward_saved_workspace_size", B, T, d, d_ff, C, k, dtype)


def layer_launches(B, T, dtype: int) -> int:
    return int(load().ipttt_layer_launches(B, T, dtype))


def _ptr(t):
    return c_vp(t.data_ptr()) if t is not None else c_vp(0)


def _need(t: torch.Tensor, name: str, shape, dtype, device):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if t.dtype != dtype:
        raise TypeError(f"{name} has dtype {t.dtype}, expected {dtype}")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


class Context:
    """An ipttt context bound to a CUDA device and (by default) torch's current stream."""

    def __init__(self, device: int | torch.device = 0, stream: torch.cuda.Stream | None = None):
        self.lib = load()
        dev = torch.device("cuda", device) if isinstance(device, int) else torch.device(device)
        self.device = dev
        self.stream = stream if stream is not None else torch.cuda.current_stream(dev)
        h = c_vp(0)
        st = self.lib.ipttt_create(ctypes.byref(h), dev.index or 0, c_vp(self.stream.cuda_stream))
        if st != IPTTT_OK:
            raise IptttError(st, "ipttt_create failed")
        self.h = h
        self._ws = None

    def close(self):
        if getattr(self, "h", None) is not None and self.h.value:
            self.lib.ipttt_destroy(self.h)
            self.h = c_vp(0)

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def _check(self, st: int, what: str):
        if st != IPTTT_OK:
            raise IptttError(st, f"{what}: {self.lib.ipttt_last_error(self.h).decode()}")

    def set_stream(self, stream: torch.cuda.Stream):
        self.stream = stream
        self._check(self.lib.ipttt_set_stream(self.h, c_vp(stream.cuda_stream)), "set_stream")

    def set_target_shift(self, shift: int):
        self._check(self.lib.ipttt_set_target_shift(self.h, int(shift)), "set_target_shift")

    def set_fused_target(self, enable: bool):
        self._check(self.lib.ipttt_set_fused_target(self.h, 1 if enable else 0), "set_fused_target")

    def set_fused_tail(self, enable: bool):
        self._check(self.lib.ipttt_set_fused_tail(self.h, 1 if enable else 0), "set_fused_tail")

    def set_apply_tiles(self, halves: int):
        """0: per call (default); 1: 256 x 256 apply tiles; 2: 256 x 512 (the fused pair kernel)."""
        self._check(self.lib.ipttt_set_apply_tiles(self.h, int(halves)), "set_apply_tiles")

    def set_cta_pairs(self, enable: bool):
        self._check(self.lib.ipttt_set_cta_pairs(self.h, 1 if enable else 0), "set_cta_pairs")

    def set_wait_limit_ns(self, ns: int):
        self._check(self.lib.ipttt_set_wait_limit_ns(self.h, int(ns)), "set_wait_limit_ns")

    def sync(self) -> int:
        """Wait for the stream and return the device status (0 = OK); raises on CUDA errors."""
        st = self.lib.ipttt_sync(self.h)
        if st not in (IPTTT_OK, 5):
            self._check(st, "sync")
        return st

    def last_error(self) -> str:
        return self.lib.ipttt_last_error(self.h).decode()

    @property
    def sm_count(self) -> int:
        return int(self.lib.ipttt_sm_count(self.h))

    def workspace(self, B, T, d, d_ff, C, k, dtype: int, host: bool = False) -> torch.Tensor:
        n = workspace_size(B, T, d, d_ff, C, k, dtype, host)
        if self._ws is None or self._ws.numel() < n:
            self._ws = torch.empty(max(n, 256), dtype=torch.uint8, device=self.device)
        return self._ws

    # ------------------------------------------------------------------ the layer
    def layer_forward(self, H, X0, W_gate, W_up, W_down0, W_target, conv_w, C: int, eta: float,
                      O=None, W_final=None, workspace=None):
        """O [B,T,d] and the final fast weight W_final [B,d,d_ff] (fp32) of the layer."""
        B, T, d = H.shape
        f = W_gate.shape[0]
        k = conv_w.shape[1]
        dt, dev = H.dtype, self.device
        for t, n, s in ((H, "H", (B, T, d)), (X0, "X0", (B, T, d)), (W_gate, "W_gate", (f, d)),
                        (W_up, "W_up", (f, d)), (W_down0, "W_down0", (d, f)), (conv_w, "conv_w", (d, k))):
            _need(t, n, s, dt, dev)
        if W_target is not None:
            _need(W_target, "W_target", (d, d), dt, dev)
        code = dtype_code(dt)
        if O is None:
            O = torch.empty((B, T, d), dtype=dt, device=dev)
        if W_final is None:
            W_final = torch.empty((B, d, f), dtype=torch.float32, device=dev)
        _need(O, "O", (B, T, d), dt, dev)
        _need(W_final, "W_final", (B, d, f), torch.float32, dev)
        ws = workspace if workspace is not None else self.workspace(B, T, d, f, C, k, code)
        st = self.lib.ipttt_layer_forward(self.h, _ptr(H), _ptr(X0), _ptr(W_gate), _ptr(W_up), _ptr(W_down0),
                                          _ptr(W_target) if W_target is not None else c_vp(0), _ptr(conv_w), B, T, d, f, C, k, float(eta), code,
                                          _ptr(O), _ptr(W_final), _ptr(ws), ws.numel() * ws.element_size())
        self._check(st, "layer_forward")
        return O, W_final

    def layer_backward(self, H, X0, W_gate, W_up, W_down0, W_target, conv_w, C: int, eta: float, dO,
                       dW_final=None, workspace=None):
        """Gradients of the layer for upstream gradients dO [B,T,d] (and dW_final [B,d,d_ff] fp32,
        None = zero).  Returns a dict: H, X0 (the activations' dtype) and W_gate, W_up, W_down0,
        W_target (None without a projection), conv_w (fp32, summed over the batch)."""
        B, T, d = H.shape
        f = W_gate.shape[0]
        k = conv_w.shape[1]
        dt, dev = H.dtype, self.device
        for t, n, s in ((H, "H", (B, T, d)), (X0, "X0", (B, T, d)), (W_gate, "W_gate", (f, d)),
                        (W_up, "W_up", (f, d)), (W_down0, "W_down0", (d, f)), (conv_w, "conv_w", (d, k)),
                        (dO, "dO", (B, T, d))):
            _need(t, n, s, dt, dev)
        if W_target is not None:
            _need(W_target, "W_target", (d, d), dt, dev)
        if dW_final is not None:
            _need(dW_final, "dW_final", (B, d, f), torch.float32, dev)
        code = dtype_code(dt)
        g = self._grad_buffers(B, T, d, f, k, dt, W_target is not None)
        if workspace is None:
            n = backward_workspace_size(B, T, d, f, C, k, code)
            workspace = torch.empty(max(n, 256), dtype=torch.uint8, device=dev)
        st = self.lib.ipttt_layer_backward(
            self.h, _ptr(H), _ptr(X0), _ptr(W_gate), _ptr(W_up), _ptr(W_down0), _ptr(W_target), _ptr(conv_w),
            B, T, d, f, C, k, float(eta), code, _ptr(dO), _ptr(dW_final), _ptr(g["H"]), _ptr(g["X0"]),
            _ptr(g["W_gate"]), _ptr(g["W_up"]), _ptr(g["W_down0"]), _ptr(g["W_target"]), _ptr(g["conv_w"]),
            _ptr(workspace), workspace.numel() * workspace.element_size())
        self._check(st, "layer_backward")
        return g

    def layer_forward_train(self, H, X0, W_gate, W_up, W_down0, W_target, conv_w, C: int, eta: float, O=None,
                            W_final=None, saved=None):
        """layer_forward that also fills a saved-activation buffer for layer_backward_saved.
        Returns (O, W_final, saved)."""
        B, T, d = H.shape
        f = W_gate.shape[0]
        k = conv_w.shape[1]
        dt, dev = H.dtype, self.device
        for t, n, s in ((H, "H", (B, T, d)), (X0, "X0", (B, T, d)), (W_gate, "W_gate", (f, d)),
                        (W_up, "W_up", (f, d)), (W_down0, "W_down0", (d, f)), (conv_w, "conv_w", (d, k))):
            _need(t, n, s, dt, dev)
        if W_target is not None:
            _need(W_target, "W_target", (d, d), dt, dev)
        code = dtype_code(dt)
        O = O if O is not None else torch.empty((B, T, d), dtype=dt, device=dev)
        W_final = W_final if W_final is not None else torch.empty((B, d, f), dtype=torch.float32, device=dev)
        if saved is None:
            saved = torch.empty(max(saved_size(B, T, d, f, C, k, code), 256), dtype=torch.uint8, device=dev)
        st = self.lib.ipttt_layer_forward_train(self.h, _ptr(H), _ptr(X0), _ptr(W_gate), _ptr(W_up), _ptr(W_down0),
                                                _ptr(W_target), _ptr(conv_w), B, T, d, f, C, k, float(eta), code,
                                                _ptr(O), _ptr(W_final), _ptr(saved),
                                                saved.numel() * saved.element_size())
        self._check(st, "layer_forward_train")
        return O, W_final, saved

    def layer_backward_saved(self, H, X0, W_gate, W_up, W_target, conv_w, C: int, eta: float, saved, dO,
                             dW_final=None, workspace=None):
        """Gradients from a buffer filled by layer_forward_train (which this call overwrites in part).
        Returns the dict of layer_backward."""
        B, T, d = H.shape
        f = W_gate.shape[0]
        k = conv_w.shape[1]
        dt, dev = H.dtype, self.device
        for t, n, s in ((H, "H", (B, T, d)), (X0, "X0", (B, T, d)), (W_gate, "W_gate", (f, d)),
                        (W_up, "W_up", (f, d)), (conv_w, "conv_w", (d, k)), (dO, "dO", (B, T, d))):
            _need(t, n, s, dt, dev)
        if W_target is not None:
            _need(W_target, "W_target", (d, d), dt, dev)
        if dW_final is not None:
            _need(dW_final, "dW_final", (B, d, f), torch.float32, dev)
        code = dtype_code(dt)
        g = self._grad_buffers(B, T, d, f, k, dt, W_target is not None)
        if workspace is None:
            n = backward_saved_workspace_size(B, T, d, f, C, k, code)
            workspace = torch.empty(max(n, 256), dtype=torch.uint8, device=dev)
        st = self.lib.ipttt_layer_backward_saved(
            self.h, _ptr(H), _ptr(X0), _ptr(W_gate), _ptr(W_up), _ptr(W_target), _ptr(conv_w), B, T, d, f, C, k,
            float(eta), code, _ptr(saved), saved.numel() * saved.element_size(), _ptr(dO), _ptr(dW_final),
            _ptr(g["H"]), _ptr(g["X0"]), _ptr(g["W_gate"]), _ptr(g["W_up"]), _ptr(g["W_down0"]), _ptr(g["W_target"]),
            _ptr(g["conv_w"]), _ptr(workspace), workspace.numel() * workspace.element_size())
        self._check(st, "layer_backward_saved")
        return g

    def _grad_buffers(self, B, T, d, f, k, dt, with_target: bool) -> dict:
        dev = self.device
        f32 = dict(dtype=torch.float32, device=dev)
        return {"H": torch.empty((B, T, d), dtype=dt, device=dev), "X0": torch.empty((B, T, d), dtype=dt, device=dev),
                "W_gate": torch.empty((f, d), **f32), "W_up": torch.empty((f, d), **f32),
                "W_down0": torch.empty((d, f), **f32),
                "W_target": torch.empty((d, d), **f32) if with_target else None,
                "conv_w": torch.empty((d, k), **f32)}

    def layer_totals(self, H, X0, W_gate, W_up, W_target, conv_w, X0_halo, C: int, eta: float, saved=None, S=None):
        """Step 1 of the three-step scheme on a range of tokens: (S, saved), S [B,d,d_ff] fp32 the
        range's update total (from zero), saved holding the range's Z and V for layer_apply_saved."""
        B, T, d = H.shape
        f = W_gate.shape[0]
        k = conv_w.shape[1]
        dt, dev = H.dtype, self.device
        for t, n, s in ((H, "H", (B, T, d)), (X0, "X0", (B, T, d)), (W_gate, "W_gate", (f, d)),
                        (W_up, "W_up", (f, d)), (conv_w, "conv_w", (d, k))):
            _need(t, n, s, dt, dev)
        if W_target is not None:
            _need(W_target, "W_target", (d, d), dt, dev)
        if X0_halo is not None:
            _need(X0_halo, "X0_halo", (B, k - 1, d), dt, dev)
        code = dtype_code(dt)
        S = S if S is not None else torch.empty((B, d, f), dtype=torch.float32, device=dev)
        if saved is None:
            saved = torch.empty(max(saved_size(B, T, d, f, C, k, code), 256), dtype=torch.uint8, device=dev)
        st = self.lib.ipttt_layer_totals(self.h, _ptr(H), _ptr(X0), _ptr(W_gate), _ptr(W_up), _ptr(W_target),
                                         _ptr(conv_w), _ptr(X0_halo if X0_halo is None or X0_halo.numel() else None),
                                         B, T, d, f, C, k, float(eta), code, _ptr(S), _ptr(saved),
                                         saved.numel() * saved.element_size())
        self._check(st, "layer_totals")
        return S, saved

    def layer_apply_saved(self, W_init, T: int, C: int, saved, dtype, O=None, W_final=None):
        """Step 3 on the range whose Z and V layer_totals saved: (O [B,T,d], W_final [B,d,d_ff] fp32)
        from each sequence's starting state W_init [B,d,d_ff] fp32."""
        B, d, f = W_init.shape
        dev = self.device
        _need(W_init, "W_init", (B, d, f), torch.float32, dev)
        O = O if O is not None else torch.empty((B, T, d), dtype=dtype, device=dev)
        W_final = W_final if W_final is not None else torch.empty((B, d, f), dtype=torch.float32, device=dev)
        st = self.lib.ipttt_layer_apply_saved(self.h, _ptr(W_init), B, T, d, f, C, dtype_code(dtype), _ptr(saved),
                                              saved.numel() * saved.element_size(), _ptr(O), _ptr(W_final))
        self._check(st, "layer_apply_saved")
        return O, W_final

    def prefix_step(self, P_in, W_down0, S, P_out, first: int = 0, count: int | None = None):
        """Step 2, one hop: P_out = (P_in, or W_down0 broadcast when P_in is None) + S (None = 0) on
        the flattened elements [first, first + count) of the [B, d, d_ff] fp32 state P_out."""
        B, d, f = P_out.shape
        dev = self.device
        _need(P_out, "P_out", (B, d, f), torch.float32, dev)
        if P_in is not None:
            _need(P_in, "P_in", (B, d, f), torch.float32, dev)
        if S is not None:
            _need(S, "S", (B, d, f), torch.float32, dev)
        if W_down0 is not None:
            _need(W_down0, "W_down0", (d, f), W_down0.dtype, dev)
        code = dtype_code(W_down0.dtype) if W_down0 is not None else F32
        count = B * d * f - first if count is None else count
        st = self.lib.ipttt_prefix_step(self.h, _ptr(P_in), _ptr(W_down0), _ptr(S), B, d, f, code, first, count,
                                        _ptr(P_out))
        self._check(st, "prefix_step")
        return P_out

    def layer_resume(self, H, X0, W_gate, W_up, W_target, conv_w, W_state, X0_halo, C: int, eta: float,
                     O=None, W_state_out=None, X0_halo_out=None, workspace=None):
        """Continue B sequences from their fp32 state and X0 halo (None = a new sequence's zeros).

        Returns O [B,T,d], the new state [B,d,d_ff] (fp32) and the new halo [B,k-1,d]."""
        B, T, d = H.shape
        f = W_gate.shape[0]
        k = conv_w.shape[1]
        dt, dev = H.dtype, self.device
        for t, n, s in ((H, "H", (B, T, d)), (X0, "X0", (B, T, d)), (W_gate, "W_gate", (f, d)),
                        (W_up, "W_up", (f, d)), (W_target, "W_target", (d, d)), (conv_w, "conv_w", (d, k))):
            _need(t, n, s, dt, dev)
        _need(W_state, "W_state", (B, d, f), torch.float32, dev)
        if X0_halo is not None:
            _need(X0_halo, "X0_halo", (B, k - 1, d), dt, dev)
        if O is None:
            O = torch.empty((B, T, d), dtype=dt, device=dev)
        if W_state_out is None:
            W_state_out = torch.empty((B, d, f), dtype=torch.float32, device=dev)
        if X0_halo_out is None:
            X0_halo_out = torch.empty((B, k - 1, d), dtype=dt, device=dev)
        _need(O, "O", (B, T, d), dt, dev)
        _need(W_state_out, "W_state_out", (B, d, f), torch.float32, dev)
        _need(X0_halo_out, "X0_halo_out", (B, k - 1, d), dt, dev)
        code = dtype_code(dt)
        ws = workspace if workspace is not None else self.workspace(B, T, d, f, C, k, code)
        st = self.lib.ipttt_layer_forward_resume(
            self.h, _ptr(H), _ptr(X0), _ptr(W_gate), _ptr(W_up), _ptr(W_target), _ptr(conv_w), _ptr(W_state),
            _ptr(X0_halo) if X0_halo is not None else c_vp(0), B, T, d, f, C, k, float(eta), code, _ptr(O),
            _ptr(W_state_out), _ptr(X0_halo_out) if X0_halo_out.numel() else c_vp(0), _ptr(ws),
            ws.numel() * ws.element_size())
        self._check(st, "layer_resume")
        return O, W_state_out, X0_halo_out

    def layer_forward_host(self, H_host, X0_host, W_gate, W_up, W_down0, W_target, conv_w, C: int, eta: float,
                           O_host, W_final_host, workspace=None):
        """The layer with H, X0, O, W_final in (pinned) host memory; asynchronous until sync()."""
        B, T, d = H_host.shape
        f = W_gate.shape[0]
        k = conv_w.shape[1]
        dt, dev = W_gate.dtype, self.device
        for t, n, s in ((W_gate, "W_gate", (f, d)), (W_up, "W_up", (f, d)), (W_down0, "W_down0", (d, f)),
                        (W_target, "W_target", (d, d)), (conv_w, "conv_w", (d, k))):
            _need(t, n, s, dt, dev)
        cpu = torch.device("cpu")
        _need(H_host, "H_host", (B, T, d), dt, cpu)
        _need(X0_host, "X0_host", (B, T, d), dt, cpu)
        _need(O_host, "O_host", (B, T, d), dt, cpu)
        _need(W_final_host, "W_final_host", (B, d, f), torch.float32, cpu)
        code = dtype_code(dt)
        ws = workspace if workspace is not None else self.workspace(B, T, d, f, C, k, code, host=True)
        st = self.lib.ipttt_layer_forward_host(self.h, _ptr(H_host), _ptr(X0_host), _ptr(W_gate), _ptr(W_up),
                                               _ptr(W_down0), _ptr(W_target), _ptr(conv_w), B, T, d, f, C, k,
                                               float(eta), code, _ptr(O_host), _ptr(W_final_host), _ptr(ws),
                                               ws.numel() * ws.element_size())
        self._check(st, "layer_forward_host")
        return O_host, W_final_host

    def state_weight(self, W_state, dtype, W=None):
        """The chunk weight from an fp32 state [B, d, d_ff]: W_state rounded to `dtype`."""
        B, d, f = W_state.shape
        _need(W_state, "W_state", (B, d, f), torch.float32, self.device)
        W = W if W is not None else torch.empty((B, d, f), dtype=dtype, device=self.device)
        _need(W, "W", (B, d, f), dtype, self.device)
        self._check(self.lib.ipttt_state_weight(self.h, _ptr(W_state), B, d, f, dtype_code(dtype), _ptr(W)),
                    "state_weight")
        return W

    def decode_step(self, H, W_gate, W_up, W_cur, X0=None, H_buf=None, X0_buf=None, pos: int = 0, O=None, Z=None):
        """A decode step (ipttt_decode_step): (O [B,m,d], Z [B,m,d_ff]) for m (1..8) new tokens H
        [B,m,d] of each sequence, applied with each sequence's chunk weight W_cur [B,d,d_ff].  With
        the chunk buffers H_buf and X0_buf [B,C,d], H and X0 [B,m,d] are also stored at tokens
        pos.. of the buffers."""
        B, m, d = H.shape
        f = W_gate.shape[0]
        dt, dev = H.dtype, self.device
        _need(H, "H", (B, m, d), dt, dev)
        for t, n, shp in ((W_gate, "W_gate", (f, d)), (W_up, "W_up", (f, d)), (W_cur, "W_cur", (B, d, f))):
            _need(t, n, shp, dt, dev)
        C = 0
        if H_buf is not None or X0_buf is not None:
            C = H_buf.shape[1]
            _need(H_buf, "H_buf", (B, C, d), dt, dev)
            _need(X0_buf, "X0_buf", (B, C, d), dt, dev)
            _need(X0, "X0", (B, m, d), dt, dev)
        O = O if O is not None else torch.empty((B, m, d), dtype=dt, device=dev)
        Z = Z if Z is not None else torch.empty((B, m, f), dtype=dt, device=dev)
        st = self.lib.ipttt_decode_step(self.h, _ptr(H), _ptr(X0), _ptr(W_gate), _ptr(W_up), _ptr(W_cur), B, m, d, f,
                                        dtype_code(dt), _ptr(Z), _ptr(O), _ptr(H_buf), _ptr(X0_buf), C, pos)
        self._check(st, "decode_step")
        return O, Z

    # ------------------------------------------------------------------ the steps
    def swiglu(self, H2d, W_gate, W_up, Z=None):
        rows, d = H2d.shape
        f = W_gate.shape[0]
        dt, dev = H2d.dtype, self.device
        _need(H2d, "H", (rows, d), dt, dev)
        _need(W_gate, "W_gate", (f, d), dt, dev)
        _need(W_up, "W_up", (f, d), dt, dev)
        if Z is None:
            Z = torch.empty((rows, f), dtype=dt, device=dev)
        _need(Z, "Z", (rows, f), dt, dev)
        self._check(self.lib.ipttt_swiglu(self.h, _ptr(H2d), _ptr(W_gate), _ptr(W_up), rows, d, f, dtype_code(dt),
                                          _ptr(Z)), "swiglu")
        return Z

    def target(self, X0, conv_w, W_target, scale: float = 1.0, V=None, Y=None):
        B, T, d = X0.shape
        k = conv_w.shape[1]
        dt, dev = X0.dtype, self.device
        _need(X0, "X0", (B, T, d), dt, dev)
        _need(conv_w, "conv_w", (d, k), dt, dev)
        _need(W_target, "W_target", (d, d), dt, dev)
        if V is None:
            V = torch.empty((B, T, d), dtype=dt, device=dev)
        if Y is None:
            Y = torch.empty((B, T, d), dtype=dt, device=dev)
        self._check(self.lib.ipttt_target(self.h, _ptr(X0), _ptr(conv_w), _ptr(W_target), B, T, d, k, float(scale),
                                          dtype_code(dt), _ptr(Y), _ptr(V)), "target")
        return V, Y

    def chunk_state(self, V, Z, W_down0, C: int, W_eff=None, W_final=None):
        B, T, d = V.shape
        f = Z.shape[2]
        n = (T + C - 1) // C
        dt, dev = V.dtype, self.device
        _need(V, "V", (B, T, d), dt, dev)
        _need(Z, "Z", (B, T, f), dt, dev)
        _need(W_down0, "W_down0", (d, f), dt, dev)
        if W_eff is None:
            W_eff = torch.empty((B, n, d, f), dtype=dt, device=dev)
        if W_final is None:
            W_final = torch.empty((B, d, f), dtype=torch.float32, device=dev)
        self._check(self.lib.ipttt_chunk_state(self.h, _ptr(V), _ptr(Z), _ptr(W_down0), B, T, d, f, C,
                                               dtype_code(dt), _ptr(W_eff), _ptr(W_final)), "chunk_state")
        return W_eff, W_final

    def chunk_apply(self, Z, W_eff, C: int, O=None):
        B, T, f = Z.shape
        d = W_eff.shape[2]
        n = (T + C - 1) // C
        dt, dev = Z.dtype, self.device
        _need(Z, "Z", (B, T, f), dt, dev)
        _need(W_eff, "W_eff", (B, n, d, f), dt, dev)
        if O is None:
            O = torch.empty((B, T, d), dtype=dt, device=dev)
        self._check(self.lib.ipttt_chunk_apply(self.h, _ptr(Z), _ptr(W_eff), B, T, d, f, C, dtype_code(dt),
                                               _ptr(O)), "chunk_apply")
        return O

    # ------------------------------------------------------------------ measurement
    def timing_begin(self):
        self._check(self.lib.ipttt_timing_begin(self.h), "timing_begin")

    def timing_read(self):
        """Per-stage summed device ms, number of timed calls, kernels those calls launched."""
        ms = (ctypes.c_double * len(STAGES))()
        calls, launches = c_i64(0), c_i64(0)
        self._check(self.lib.ipttt_timing_read(self.h, ms, ctypes.byref(calls), ctypes.byref(launches)),
                    "timing_read")
        return dict(zip(STAGES, list(ms))), calls.value, launches.value

    def selftest_wait_timeout(self):
        self._check(self.lib.ipttt_selftest_wait_timeout(self.h), "selftest_wait_timeout")


DECODE_MAX_TOKENS = 8  # tokens per sequence that one ipttt_decode_step takes


class StreamingLayer:
    """Keeps the per-sequence fast-weight state and conv halo of B sequences across calls.

    step() takes any number of tokens per call (one token at a time for decoding):
      * whole chunks starting at a chunk boundary run through the resumable layer;
      * tokens of a chunk that is not complete yet are applied at once with the weight at the
        chunk's start, and their inputs are buffered; when the chunk completes, its update is
        committed by running the resumable layer over the buffered chunk (the C-token buffer of
        a decode loop).  Up to 8 such tokens per call go through ipttt_decode_step (weight-streaming
        decode rows); more, or all of them with exact=True, through the SwiGLU step and the chunk
        apply, the tensor-core kernels of the chunked call.
    The state after every complete chunk equals that of one call over the whole sequence bit for
    bit, and so do the outputs of whole chunks and, with exact=True, every output; the decode
    rows agree with them to rounding.  flush() commits a final partial chunk, after which
    `state` is the final W_down of the whole sequence.  Buffers only: all compute runs in the
    library.
    """

    def __init__(self, ctx: Context, W_gate, W_up, W_down0, W_target, conv_w, B: int, C: int, eta: float,
                 exact: bool = False):
        self.ctx, self.C, self.eta, self.B, self.exact = ctx, C, eta, B, exact
        self.W_gate, self.W_up, self.W_target, self.conv_w = W_gate, W_up, W_target, conv_w
        d, f = W_down0.shape
        k = conv_w.shape[1]
        dt, dev = W_down0.dtype, W_down0.device
        self.d, self.f, self.dtype = d, f, dt
        empty = torch.empty((B, 0, d), dtype=dt, device=dev)
        # an empty call leaves every sequence's state at W_down0 (fp32)
        _, self.state = ctx.layer_forward(empty, empty, W_gate, W_up, W_down0, W_target, conv_w, C, eta)
        self.state = self.state.clone()
        self.halo = torch.zeros((B, k - 1, d), dtype=dt, device=dev)
        self._halo_next = torch.empty_like(self.halo)
        self.W_cur = torch.empty((B, d, f), dtype=dt, device=dev)  # the weight of the current chunk
        self._w_cur_ok = False  # W_cur holds the weight of the current state
        self.pending = 0  # tokens of the current chunk already seen
        self._pend_H = torch.empty((B, C, d), dtype=dt, device=dev)
        self._pend_X = torch.empty((B, C, d), dtype=dt, device=dev)

    def _resume(self, H, X0, O=None):
        O, self.state, self._halo_next = self.ctx.layer_resume(
            H, X0, self.W_gate, self.W_up, self.W_target, self.conv_w, self.state, self.halo, self.C, self.eta,
            O=O, W_state_out=self.state, X0_halo_out=self._halo_next)
        self.halo, self._halo_next = self._halo_next, self.halo
        self._w_cur_ok = False
        return O

    def _commit_pending(self):
        n = self.pending
        self._resume(self._pend_H[:, :n].contiguous(), self._pend_X[:, :n].contiguous())
        self.pending = 0

    def step(self, H, X0, O=None):
        B, n, d = H.shape
        outs, pos = [], 0
        while pos < n:
            if self.pending == 0 and n - pos >= self.C:
                m = (n - pos) // self.C * self.C
                outs.append(self._resume(H[:, pos:pos + m].contiguous(), X0[:, pos:pos + m].contiguous()))
                pos += m
                continue
            m = min(self.C - self.pending, n - pos)
            if not self._w_cur_ok:  # first tokens of a chunk: its weight, from the state
                self.ctx.state_weight(self.state, self.dtype, self.W_cur)
                self._w_cur_ok = True
            h = H[:, pos:pos + m].contiguous()
            if self.exact or m > DECODE_MAX_TOKENS:
                Z = self.ctx.swiglu(h.view(B * m, d), self.W_gate, self.W_up)
                outs.append(self.ctx.chunk_apply(Z.view(B, m, self.f), self.W_cur.view(B, 1, d, self.f), self.C))
                self._pend_H[:, self.pending:self.pending + m] = h
                self._pend_X[:, self.pending:self.pending + m] = X0[:, pos:pos + m]
            else:
                O_t, _ = self.ctx.decode_step(h, self.W_gate, self.W_up, self.W_cur, X0[:, pos:pos + m].contiguous(),
                                              self._pend_H, self._pend_X, self.pending)
                outs.append(O_t)
            self.pending += m
            pos += m
            if self.pending == self.C:
                self._commit_pending()
        out = outs[0] if len(outs) == 1 else torch.cat(outs, dim=1)
        if O is not None:
            O.copy_(out)
            return O
        return out

    def flush(self):
        """Commit the update of a final partial chunk (the stream ends inside a chunk)."""
        if self.pending:
            self._commit_pending()
