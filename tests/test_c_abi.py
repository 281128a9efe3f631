"""The C ABI as a C caller sees it: a plain C99 translation unit is compiled against
include/moe_gb300.h with gcc, linked with libmoe_gb300.so and run.  It calls only the
host-side entry points, so no GPU is needed."""
import os
import shutil
import subprocess

import pytest

import mixture_experts_grouped_align_gb300 as moe

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_plain_c_caller_compiles_links_and_runs(tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    lib = moe.build()
    exe = str(tmp_path / "abi_host_check")
    src = os.path.join(ROOT, "tests", "c", "abi_host_check.c")
    cmd = [cc, "-std=c99", "-Wall", "-Werror", "-pedantic", "-I", os.path.join(ROOT, "include"), src,
           "-o", exe, "-L", os.path.dirname(lib), "-lmoe_gb300", "-Wl,-rpath," + os.path.dirname(lib)]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.strip().endswith("ok: 0 failure(s)"), r.stdout
