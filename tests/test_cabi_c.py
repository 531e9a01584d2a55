"""The C ABI from a plain C99 program (CPU only): tests/c/abi_host.c includes only
include/gcs_attn.h, links libgcs_attn.so, and checks validation and workspace sizes without
addressing device memory or launching anything."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_c_program_uses_the_abi(tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    from gated_causal_softmax_gb300 import build

    lib = build.build()
    libdir = os.path.dirname(lib)
    exe = tmp_path / "abi_host"
    cmd = [cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
           os.path.join(ROOT, "tests", "c", "abi_host.c"), "-o", str(exe), "-L", libdir, "-lgcs_attn",
           "-Wl,-rpath," + libdir]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.strip() == "ok"
