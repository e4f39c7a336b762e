"""include/igemm.h compiles as C and a C program links against libigemm.so
and gets the documented answers from the argument checks (no GPU needed)."""

import os
import shutil
import subprocess

import pytest

import precision_integer_gemm_gb300 as pig

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CUDA_INCLUDE = "/usr/local/cuda/include"


def test_c_program_against_the_header(tmp_path):
    if not shutil.which("gcc") or not os.path.isdir(CUDA_INCLUDE):
        pytest.skip("gcc or the CUDA headers are missing")
    pig.build_library()
    lib_dir = os.path.dirname(pig.LIB_PATH)
    exe = str(tmp_path / "abi_check")
    cmd = ["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), "-I", CUDA_INCLUDE,
           os.path.join(ROOT, "tests", "c", "abi_check.c"), "-o", exe, "-L", lib_dir,
           "-l:" + os.path.basename(pig.LIB_PATH), "-Wl,-rpath," + lib_dir]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stderr
    assert r.stdout.startswith("c abi ok")
