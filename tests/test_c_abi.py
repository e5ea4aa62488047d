"""The C ABI from C: tests/c/abi_check.c is compiled as C11 against
include/ltk.h, linked against libltk.so and run (host-only entry points, no
GPU).  This shows the header is plain C and the library serves a C caller
without Python."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_c_client_compiles_links_and_runs(ltk_lib, tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    from indexer_topk_long_gb300 import library_path
    libdir = os.path.dirname(library_path())
    exe = str(tmp_path / "abi_check")
    build = subprocess.run(
        [cc, "-std=c11", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", os.path.join(ROOT, "include"),
         os.path.join(ROOT, "tests", "c", "abi_check.c"), "-o", exe, "-L", libdir, "-lltk",
         f"-Wl,-rpath,{libdir}"],
        capture_output=True, text=True)
    assert build.returncode == 0, build.stderr
    run = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert run.returncode == 0, run.stdout + run.stderr
    assert run.stdout.strip() == "abi ok"
