"""The boundary from plain C: a C program (tests/c/abi_from_c.c) allocates with cudaMalloc,
calls sb_lmhead_project through include/sb.h, and checks the results against the oracle."""
import os
import subprocess

import pytest

import oracle
from gemm_epilogue_reduction_gb300 import build as sbbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _compile(tmp_path):
    lib = sbbuild.build()
    olib = oracle.build()
    exe = str(tmp_path / "abi_from_c")
    cuda = "/usr/local/cuda"
    cmd = ["gcc", "-O1", "-std=c11", os.path.join(ROOT, "tests", "c", "abi_from_c.c"),
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(cuda, "include"),
           lib, olib, "-L", os.path.join(cuda, "lib64"), "-lcudart", "-lm",
           "-Wl,-rpath," + os.path.dirname(lib) + ":" + os.path.dirname(olib) + ":" +
           os.path.join(cuda, "lib64"), "-o", exe]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    return exe


def test_c_program_compiles_against_the_header(tmp_path):
    _compile(tmp_path)


@pytest.mark.gpu
def test_c_program_runs_the_projection(tmp_path):
    exe = _compile(tmp_path)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "C ABI ok" in r.stdout
