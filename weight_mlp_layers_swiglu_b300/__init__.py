"""In-Place TTT fast-weight SwiGLU layer for NVIDIA B300 (sm_103a).

The compute lives in libipttt.so (hand-written tcgen05/TMA kernels, C ABI in
include/ipttt.h); this package is its thin ctypes binding plus the seeded
synthetic workloads.  There is no CPU fallback.
"""
from .native import (BF16, F32, STAGES, Context, IptttError, StreamingLayer, dtype_code, exported_symbols,
                     backward_saved_workspace_size, backward_workspace_size, layer_launches, load, saved_size,
                     workspace_size)

__all__ = ["BF16", "F32", "STAGES", "Context", "IptttError", "StreamingLayer", "dtype_code", "exported_symbols",
           "backward_saved_workspace_size", "backward_workspace_size", "layer_launches", "load", "saved_size",
           "workspace_size"]
