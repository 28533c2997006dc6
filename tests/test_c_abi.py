"""The C ABI called from plain C (tests/c_abi_caller.c): no Python, no torch.

The program is compiled with gcc against include/gbconv.h and linked with
libgbconv.so, the fp64 test oracle (liboracle.so) and the CUDA runtime. On a
machine without a supported GPU it checks the validation path (a valid call
reports the unsupported device, a bad descriptor its own code); on a GB300 it
runs three convolutions through AUTO (an fp32 stem, a wide fp32 layer, a
bf16 causal conv3d) with cudaMalloc'd buffers and compares each with the
oracle.
"""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "implicit_gemm_convolution_conv_gb300")
ORACLE = os.path.join(ROOT, "oracle")
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


def _build(tmp_path):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not found")
    lib64 = os.path.join(CUDA, "lib64")
    exe = str(tmp_path / "c_abi_caller")
    cmd = ["gcc", "-std=c99", "-O2", "-I", os.path.join(ROOT, "include"),
           "-I", os.path.join(CUDA, "include"),
           os.path.join(ROOT, "tests", "c_abi_caller.c"), "-o", exe,
           "-L", PKG, "-lgbconv", "-L", ORACLE, "-loracle", "-L", lib64, "-lcudart", "-lm",
           f"-Wl,-rpath,{PKG}:{ORACLE}:{lib64}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return exe


def _run(exe):
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    return r.returncode, r.stdout + r.stderr


def test_c_caller_builds_and_validates(tmp_path):
    """Builds against the header and both libraries; without a GPU it checks
    the status codes, with one it runs the parity cases."""
    rc, out = _run(_build(tmp_path))
    assert rc == 0, out


@pytest.mark.gpu
def test_c_caller_parity_on_gpu(tmp_path):
    rc, out = _run(_build(tmp_path))
    assert rc == 0, out
    assert out.count(" ok") == 3, out
