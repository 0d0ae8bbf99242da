"""The C ABI from plain C: tests/c/abi_host.c is compiled as C99 with gcc against
include/ipttt.h, linked with libipttt.so, and run.  It makes host-only calls (no GPU), so it
shows that the header is valid C and the library usable without Python; its sizes must equal
the ones the Python binding reports."""
import os
import shutil
import subprocess

import pytest

import weight_mlp_layers_swiglu_b300 as pkg
from weight_mlp_layers_swiglu_b300 import native

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
def test_header_and_library_from_plain_c(tmp_path):
    pkg.load()
    lib = native._build.LIB_PATH
    exe = tmp_path / "abi_host"
    cmd = ["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", os.path.join(ROOT, "include"),
           os.path.join(ROOT, "tests", "c", "abi_host.c"), "-o", str(exe), lib,
           f"-Wl,-rpath,{os.path.dirname(lib)}"]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    run = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert run.returncode == 0, run.stdout + run.stderr
    lines = dict(l.split(" ", 1) for l in run.stdout.splitlines() if l.startswith(("workspace ", "saved ")))
    assert int(lines["workspace"]) == pkg.workspace_size(1, 32768, 2560, 9728, 1024, 4, pkg.BF16)
    assert int(lines["saved"]) == pkg.saved_size(1, 32768, 2560, 9728, 1024, 4, pkg.BF16)
