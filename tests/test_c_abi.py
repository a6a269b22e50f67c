"""libfd from a plain C program (tests/c/c_abi_decode.c): include/fd.h must compile as
C99 with warnings as errors, and the program must link against libfd.so alone (plus the
CUDA runtime and, for its check, the fp64 oracle).  On a GPU the program runs a decode
through fd_decode_attention, fd_decode_attention_ex and a plan, and compares every output
with the oracle itself."""
import glob
import os
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c", "c_abi_decode.c")


def _cuda_dirs():
    from decode_attention_05_gb300 import build as fd_build
    home = os.path.dirname(os.path.dirname(os.path.realpath(fd_build.nvcc())))
    libs = [p for p in [os.path.join(home, "lib64"), *glob.glob(os.path.join(home, "targets", "*", "lib"))]
            if glob.glob(os.path.join(p, "libcudart.so*"))]
    return os.path.join(home, "include"), libs[0]


def _build(tmp_path):
    from decode_attention_05_gb300 import build as fd_build
    import oracle
    fd_lib = fd_build.build()
    oracle_lib = oracle.build()
    inc, cudalib = _cuda_dirs()
    exe = str(tmp_path / "c_abi_decode")
    lib_dirs = [os.path.dirname(fd_lib), os.path.dirname(oracle_lib), cudalib]
    cmd = ["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-O1", SRC, "-o", exe,
           "-I", os.path.join(ROOT, "include"), "-I", inc]
    for d in lib_dirs:
        cmd += ["-L", d, "-Wl,-rpath," + d]
    cmd += ["-lfd", "-lfd_oracle", "-lcudart", "-lm"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    return exe


def test_c_program_compiles_and_links(tmp_path):
    assert os.path.exists(_build(tmp_path))


@pytest.mark.gpu
def test_c_program_decodes_against_the_oracle(tmp_path):
    exe = _build(tmp_path)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "c abi ok" in r.stdout
