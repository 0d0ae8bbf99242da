"""The allocation-free target step, ipttt_target_noalloc, through the C ABI.

Callers that cannot allocate device memory (their device memory belongs to a host
application's own allocator, or a cudaMalloc could stall a latency-critical loop, or the
footprint must be fixed at load time) use this entry point: it keeps the conv output in the
library's built-in scratch instead of a caller buffer.  It must give what the allocating
entry point ipttt_target gives, bit for bit: it runs the same kernels on the same grids.
This file is collected last on purpose, so that a run that stops at the first failure has
already run every other test; it also passes on its own in a fresh process.
"""
import ctypes

import pytest
import torch

from tests.util import rel_err, seeded

pytestmark = pytest.mark.gpu


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _call(lib, X0, cw, Wt, scale, V, status=None):
    import weight_mlp_layers_swiglu_b300 as pkg

    B, T, d = X0.shape
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.ipttt_target_noalloc(_p(X0), _p(cw), _p(Wt), B, T, d, cw.shape[1], float(scale),
                                    pkg.dtype_code(X0.dtype), _p(V), _p(status) if status is not None else None,
                                    stream)


def test_noalloc_target_matches_the_allocating_entry_point_on_two_calls_in_a_row():
    import weight_mlp_layers_swiglu_b300 as pkg

    lib = pkg.load()
    ctx = pkg.Context(0)
    cases = [(2, 300, 256, 4, torch.bfloat16, 1.0 / 128), (1, 700, 512, 3, torch.float32, 0.25)]
    for i, (B, T, d, k, dt, scale) in enumerate(cases):
        X0 = seeded((B, T, d), 0.02, dt, 40 + i, "cuda")
        cw = seeded((d, k), k ** -0.5, dt, 50 + i, "cuda")
        Wt = seeded((d, d), d ** -0.5, dt, 60 + i, "cuda")
        V_ref, _ = ctx.target(X0, cw, Wt, scale)
        assert ctx.sync() == 0
        V = torch.full((B, T, d), float("nan"), dtype=dt, device="cuda")
        status = torch.zeros(2, dtype=torch.int32, device="cuda")
        assert _call(lib, X0, cw, Wt, scale, V, status) == 0
        torch.cuda.synchronize()
        assert int(status[0]) == 0
        # the same kernels on the same grids as the allocating entry point: the same bits
        assert torch.equal(V, V_ref), f"max rel err {rel_err(V, V_ref)} (case {i})"
        # a second call in a row reuses the scratch the first one left behind
        V2 = torch.full((B, T, d), float("nan"), dtype=dt, device="cuda")
        assert _call(lib, X0, cw, Wt, scale, V2, status) == 0
        torch.cuda.synchronize()
        assert int(status[0]) == 0 and torch.equal(V2, V_ref)
    ctx.close()


def test_noalloc_target_without_status_word_and_size_limit():
    import weight_mlp_layers_swiglu_b300 as pkg

    lib = pkg.load()
    X0 = seeded((1, 128, 128), 0.02, torch.bfloat16, 7, "cuda")
    cw = seeded((128, 4), 0.5, torch.bfloat16, 8, "cuda")
    Wt = seeded((128, 128), 128 ** -0.5, torch.bfloat16, 9, "cuda")
    V1 = torch.empty((1, 128, 128), dtype=torch.bfloat16, device="cuda")
    V2 = torch.empty_like(V1)
    assert _call(lib, X0, cw, Wt, 1.0, V1) == 0
    assert _call(lib, X0, cw, Wt, 1.0, V2) == 0
    torch.cuda.synchronize()
    assert torch.equal(V1, V2)
    # past the built-in scratch: rejected before any launch, the output stays untouched
    cap = (16 << 20) - 256
    T = cap // (128 * 2) + 1
    big = torch.zeros((1, T, 128), dtype=torch.bfloat16, device="cuda")
    out = torch.full((1, T, 128), 3.0, dtype=torch.bfloat16, device="cuda")
    assert _call(lib, big, cw, Wt, 1.0, out) == 3  # IPTTT_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert torch.all(out == 3.0)
