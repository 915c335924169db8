"""The C ABI used from plain C: tests/c_client.c includes only
include/fa_splitkv.h, is compiled with gcc (-std=c99 -Wall -Werror) and linked
against the shared library, and checks the host-only entry points.  CPU only."""

import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.skipif(shutil.which("gcc") is None, reason="no C compiler")
def test_c_client_compiles_links_and_runs(tmp_path):
    import split_kv_flashattention_gb300 as pkg
    if not os.path.exists(pkg.LIB_PATH):
        from split_kv_flashattention_gb300 import build
        build.build()
    libdir = os.path.dirname(pkg.LIB_PATH)
    exe = str(tmp_path / "c_client")
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror",
                    "-I", os.path.join(ROOT, "include"), os.path.join(ROOT, "tests", "c_client.c"),
                    "-L", libdir, "-lfa_splitkv", "-Wl,-rpath," + libdir, "-o", exe], check=True)
    res = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert res.returncode == 0, res.stdout + res.stderr
    assert "c client ok" in res.stdout
