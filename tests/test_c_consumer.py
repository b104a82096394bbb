"""The C ABI used from C: tests/c/consumer.c is compiled as C99 against include/gemm.h
and linked against the library, then run (host-only entry points; no GPU needed)."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib_dir():
    from dense_tiled_gemm_05_gb300 import build as gbuild
    gbuild.build()
    d = os.path.join(ROOT, "dense_tiled_gemm_05_gb300", "_lib")
    assert os.path.exists(os.path.join(d, "libgemm_gb300.so"))
    return d


def test_c_program_compiles_and_runs(lib_dir, tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    exe = tmp_path / "consumer"
    subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic",
                    "-I", os.path.join(ROOT, "include"), os.path.join(ROOT, "tests", "c", "consumer.c"),
                    "-L", lib_dir, "-lgemm_gb300", "-Wl,-rpath," + lib_dir, "-o", str(exe)],
                   check=True, capture_output=True, text=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr + r.stdout
    assert "all checks passed" in r.stdout
