"""The C ABI from plain C: `tests/c_client.c` includes only include/w4a16.h,
compiles as strict C99, links the in-tree shared library and runs the entry
points that need no GPU (no CUDA work is launched)."""
import os
import shutil
import subprocess

import pytest

import gemm_w4a16_group_gb300 as w4

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_header_compiles_as_c99_and_links(tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    w4.lib()  # builds the library if it is missing or stale
    libdir = os.path.dirname(w4.library_path())
    exe = str(tmp_path / "c_client")
    cmd = [cc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror", "-I", os.path.join(ROOT, "include"),
           os.path.join(ROOT, "tests", "c_client.c"), "-o", exe, "-L", libdir, "-lw4a16_gb300",
           "-Wl,-rpath," + libdir]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "c client ok" in r.stdout
