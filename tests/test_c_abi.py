"""The header compiles as strict C and the library links and runs from C (host-only
calls: the block manager on the vLLM post's examples). No GPU."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_c_program_uses_the_abi():
    from paged_kv_cache_02_gb300 import _build
    lib = _build.build()
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    out_dir = os.path.join(_build.BUILD, "ctest")
    os.makedirs(out_dir, exist_ok=True)
    exe = os.path.join(out_dir, "bm_example")
    libdir = os.path.dirname(lib)
    cmd = [cc, "-std=c11", "-Wall", "-Wextra", "-Werror", "-pedantic",
           "-I", os.path.join(ROOT, "include"), os.path.join(ROOT, "tests", "c", "bm_example.c"),
           "-L", libdir, "-lpa", f"-Wl,-rpath,{libdir}", "-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "FAIL" not in r.stdout and r.stdout.count("ok") >= 12
