"""Host-only checks of the C ABI (no GPU needed): the library builds, loads and exports
every entry point include/ipttt.h declares, and the host-side validation answers."""
import ctypes
import os
import re

import pytest

import weight_mlp_layers_swiglu_b300 as pkg
from weight_mlp_layers_swiglu_b300 import native

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ipttt.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ipttt_[a-z_]+)\s*\(", text)))


def test_header_declares_the_binding_surface():
    names = declared_functions()
    assert "ipttt_layer_forward" in names and "ipttt_create" in names
    assert sorted(native.exported_symbols()) == names


def test_library_exports_every_declared_symbol():
    lib = pkg.load()
    out = os.popen(f"nm -D --defined-only {native._build.LIB_PATH}").read()
    exported = set(re.findall(r" T (ipttt_[a-z_]+)", out))
    for name in declared_functions():
        assert name in exported, name
        assert hasattr(lib, name)


def test_version_and_status_strings():
    lib = pkg.load()
    assert re.match(rb"^\d+\.\d+\.\d+$", lib.ipttt_version())
    assert lib.ipttt_status_string(0) == b"IPTTT_OK"
    assert lib.ipttt_status_string(5) == b"IPTTT_ERR_TIMEOUT"


def _ws(*args):
    lib = pkg.load()
    out = ctypes.c_size_t(0)
    st = lib.ipttt_workspace_size(*args, ctypes.byref(out))
    return st, out.value


def test_workspace_size_layout():
    B, T, d, f, C, k = 2, 1000, 256, 512, 128, 4
    st, n = _ws(B, T, d, f, C, k, pkg.BF16)
    assert st == 0
    a = lambda x: (x + 255) // 256 * 256
    nch = (T + C - 1) // C
    ctr = a((B * nch + 1) * 4)
    assert n == a(B * T * d * 2) * 2 + a(B * T * f * 2) + a(B * nch * d * f * 2) + ctr
    st, n32 = _ws(B, T, d, f, C, k, pkg.F32)
    assert st == 0 and n32 == a(B * T * d * 4) * 2 + a(B * T * f * 4) + a(B * nch * d * f * 4) + ctr
    # the 4B-shaped 32k workload fits comfortably in HBM
    st, n = _ws(1, 32768, 2560, 9728, 1024, 4, pkg.BF16)
    assert st == 0 and n < 3e9


@pytest.mark.parametrize("args,code", [
    ((1, 64, 256, 512, 100, 4, 1), 2),    # bf16 needs C % 128 == 0
    ((1, 64, 256, 512, 100, 4, 0), 0),    # fp32 takes any C
    ((1, 64, 250, 512, 128, 4, 1), 2),    # d % 8
    ((1, 64, 256, 500, 128, 4, 1), 2),    # d_ff % 8
    ((1, 64, 256, 512, 128, 9, 1), 2),    # k > 8
    ((1, 64, 256, 512, 128, 0, 1), 1),    # k < 1
    ((-1, 64, 256, 512, 128, 4, 1), 1),   # negative B
    ((1, -5, 256, 512, 128, 4, 1), 1),    # negative T
    ((1, 64, 256, 512, 0, 4, 1), 1),      # C < 1
    ((1, 64, 256, 512, 128, 4, 7), 1),    # unknown dtype
    ((0, 0, 256, 512, 128, 4, 1), 0),     # empty batch is fine
])
def test_workspace_size_validation(args, code):
    st, _ = _ws(*args)
    assert st == code


def test_null_context_and_outputs_are_rejected():
    lib = pkg.load()
    assert lib.ipttt_workspace_size(1, 1, 8, 8, 1, 1, 0, None) == 1
    assert lib.ipttt_sync(None) == 1
    assert lib.ipttt_layer_forward(None, *([None] * 7), 1, 1, 8, 8, 1, 1, 0.1, 0, None, None, None, 0) == 1
    lib.ipttt_destroy(None)


def test_launch_counts():
    assert pkg.layer_launches(1, 32768, pkg.BF16) == 4
    assert pkg.layer_launches(1, 2048, pkg.F32) == 6
    assert pkg.layer_launches(3, 0, pkg.BF16) == 1
    assert pkg.layer_launches(0, 100, pkg.BF16) == 0


def _size(fn, *args):
    lib = pkg.load()
    out = ctypes.c_size_t(0)
    st = getattr(lib, fn)(*args, ctypes.byref(out))
    return st, out.value


def test_training_buffer_sizes():
    """The saved-activation buffer holds Z, [A | U], Y, V and every W_i (dtype) plus the counters;
    the backward-from-saved workspace holds only the backward's own scratch, and the recomputing
    backward's workspace is the two together."""
    B, T, d, f, C, k = 2, 1000, 256, 512, 128, 4
    a = lambda x: (x + 255) // 256 * 256
    n = (T + C - 1) // C
    st, saved = _size("ipttt_saved_size", B, T, d, f, C, k, pkg.BF16)
    assert st == 0
    assert saved == a(B * T * f * 2) + a(B * T * 2 * f * 2) + 2 * a(B * T * d * 2) + a(B * n * d * f * 2) + a(
        (B * n + 1) * 4)
    st, scratch = _size("ipttt_backward_saved_workspace_size", B, T, d, f, C, k, pkg.BF16)
    strips = B * ((T + 63) // 64)
    assert st == 0 and scratch == 2 * a(B * T * d * 2) + a(B * n * d * f * 2) + a(B * d * f * 4) + a(strips * d * k * 4)
    st, full = _size("ipttt_backward_workspace_size", B, T, d, f, C, k, pkg.BF16)
    assert st == 0 and full == saved + scratch
    # fp32 adds dZ to the scratch
    st, scratch32 = _size("ipttt_backward_saved_workspace_size", B, T, d, f, C, k, pkg.F32)
    assert st == 0 and scratch32 == a(B * T * f * 4) + 2 * a(B * T * d * 4) + a(B * n * d * f * 4) + a(
        B * d * f * 4) + a(strips * d * k * 4)
    assert _size("ipttt_saved_size", 1, 64, 250, 512, 128, 4, pkg.BF16)[0] == 2  # d % 8


def test_host_workspace_holds_one_piece():
    """The host-buffer entry's workspace: the layer workspace for one piece (4096 tokens, a
    multiple of C) plus whole H, X0, O, the fp32 state and two halos."""
    B, T, d, f, C, k = 1, 32768, 2560, 9728, 1024, 4
    st, host = _size("ipttt_host_workspace_size", B, T, d, f, C, k, pkg.BF16)
    st2, piece = _size("ipttt_workspace_size", B, 4096, d, f, C, k, pkg.BF16)
    a = lambda x: (x + 255) // 256 * 256
    assert st == 0 and st2 == 0
    assert host == piece + 3 * a(B * T * d * 2) + a(B * d * f * 4) + 2 * a(B * (k - 1) * d * 2)



def _declarations():
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    for m in re.finditer(r"([A-Za-z_][\w \*]*?)\b(ipttt_[a-z_]+)\s*\(([^)]*)\)\s*;", text):
        params = [" ".join(p.split()) for p in m.group(3).split(",")]
        yield m.group(2), m.group(1).strip(), [] if params == ["void"] else params


def _c_kind(decl: str):
    """The kind of value a C parameter (with its name) or return type carries."""
    stars = decl.count("*")
    words = [w for w in decl.replace("*", " ").split() if w != "const"]
    base = words[0]
    if stars >= 2:
        return "ptrptr"
    if stars == 1:
        return {"char": "char_p", "size_t": "size_p"}.get(base, "ptr")
    return {"int64_t": "i64", "uint64_t": "u64", "int": "i32", "ipttt_dtype": "i32", "ipttt_status": "i32",
            "float": "f32", "double": "f64", "size_t": "size", "void": None}[base]


def _ctypes_kind(t):
    if t is None:
        return None
    if t is ctypes.c_char_p:
        return "char_p"
    if t is ctypes.c_void_p:
        return "ptr"
    if t is ctypes.POINTER(ctypes.c_void_p):
        return "ptrptr"
    if t is ctypes.POINTER(ctypes.c_size_t):
        return "size_p"
    if isinstance(t, type) and issubclass(t, ctypes._Pointer):
        return "ptr"
    return {ctypes.c_int64: "i64", ctypes.c_uint64: "u64", ctypes.c_int: "i32", ctypes.c_float: "f32",
            ctypes.c_double: "f64", ctypes.c_size_t: "size"}[t]


def test_binding_signatures_match_the_header():
    """Every argument the binding marshals has the width and kind the header declares, so a
    shifted or missing argument fails here rather than on the device."""
    sigs = native._SIGNATURES
    decls = {name: (ret, params) for name, ret, params in _declarations()}
    assert set(sigs) <= set(decls)
    for name, (restype, argtypes) in sigs.items():
        ret, params = decls[name]
        want = [_c_kind(p) for p in params]
        got = [_ctypes_kind(t) for t in argtypes]
        assert len(got) == len(want), (name, len(got), len(want))
        for i, (g, w) in enumerate(zip(got, want)):
            # A size_t* result may be passed as a plain address; size_t and uint64_t are one
            # ctypes type on this platform.
            w = "u64" if w == "size" else w
            g = "u64" if g == "size" else g
            assert g == w or (w == "size_p" and g == "ptr"), (name, i, params[i], g)
        assert _ctypes_kind(restype) == _c_kind(ret), (name, ret)
