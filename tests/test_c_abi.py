"""The C ABI used from a plain C99 program (no C++, no Python in the call path): the header
compiles as C, the program links against the library, and -- on a GPU -- computes a known
result under every schedule."""
import os
import shutil
import subprocess

import pytest

from sm_constrained_persistent_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


def _compile(tmp_path):
    if shutil.which("gcc") is None:
        pytest.skip("no C compiler")
    _build.build()
    exe = str(tmp_path / "c_abi_check")
    lib_dir = os.path.dirname(_build.LIB_PATH)
    cmd = ["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror",
           os.path.join(ROOT, "tests", "c_abi_check.c"), "-o", exe,
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(CUDA, "include"),
           "-L", lib_dir, "-L", os.path.join(CUDA, "lib64"), "-lskgemm", "-lcudart",
           "-Wl,-rpath," + lib_dir + ":" + os.path.join(CUDA, "lib64")]
    subprocess.run(cmd, check=True)
    return exe


def test_header_is_strict_c99(tmp_path):
    if shutil.which("gcc") is None:
        pytest.skip("no C compiler")
    src = tmp_path / "h.c"
    src.write_text('#include "sk_gemm.h"\nint main(void) { return SK_MODE_AUTO - 4; }\n')
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-fsyntax-only",
                    "-I", os.path.join(ROOT, "include"), str(src)], check=True)


def test_c_program_builds_and_runs_the_host_calls(tmp_path):
    import torch
    if torch.cuda.is_available():
        pytest.skip("covered by the GPU test")
    exe = _compile(tmp_path)
    r = subprocess.run([exe], capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr


@pytest.mark.gpu
def test_c_program_computes_the_addmm_under_every_schedule(tmp_path):
    exe = _compile(tmp_path)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "passed" in r.stdout
