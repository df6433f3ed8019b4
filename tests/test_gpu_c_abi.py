"""A plain C caller of the C ABI (tests/c_abi_forward.c): cudaMalloc'd buffers, the
workspace sized and initialised through the library, one moe_forward, y checked
against the fp64 oracle's C library. Built here with nvcc as the compiler driver
against libmoe.so and oracle/liboracle.so, then run as its own process."""
from __future__ import annotations

import os
import shutil
import subprocess

import pytest
import torch

import oracle
from moe_expert_router_gb300 import binding as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.gpu
def test_c_caller_forward(tmp_path):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    B.load()                            # raises when libmoe.so is missing: there is no fallback
    pkg_dir = os.path.dirname(os.path.abspath(B.LIB_PATH))
    oracle_dir = os.path.dirname(oracle.build())
    nvcc = os.environ.get("NVCC") or shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    exe = str(tmp_path / "c_abi_forward")
    cmd = [nvcc, "-O2", "-I", os.path.join(ROOT, "include"), os.path.join(ROOT, "tests", "c_abi_forward.c"),
           "-o", exe, "-L", pkg_dir, "-lmoe", "-L", oracle_dir, "-loracle",
           "-Xlinker", "-rpath", "-Xlinker", f"{pkg_dir}:{oracle_dir}", "-lm"]
    build = subprocess.run(cmd, capture_output=True, text=True)
    assert build.returncode == 0, build.stderr
    run = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert run.returncode == 0, run.stdout + run.stderr
    assert "relative Frobenius error" in run.stdout
