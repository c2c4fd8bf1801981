"""tcgen05 building blocks on the GPU, one CTA each, against CPU products:
the Q K^T shape (K-major SW128 operands), the P V shape with an MN-major B
operand, and P V with the A operand in tensor memory."""
import ctypes
import os
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "native", "tcgen05_selftest.cu")
OUT = os.path.join(HERE, "native", "_build", "libfia_selftest.so")


def _build():
    os.makedirs(os.path.dirname(OUT), exist_ok=True)
    if not os.path.exists(OUT) or os.path.getmtime(OUT) < max(os.path.getmtime(SRC), os.path.getmtime(
            os.path.join(HERE, "..", "attention_fia_prefill_gb300", "csrc", "ptx.cuh"))):
        cmd = ["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-std=c++17", "-shared",
               "-Xcompiler", "-fPIC", "-cudart", "shared", SRC, "-o", OUT]
        subprocess.run(cmd, check=True)
    lib = ctypes.CDLL(OUT)
    lib.fia_selftest_run.argtypes = [ctypes.c_int]
    lib.fia_selftest_run.restype = ctypes.c_double
    return lib


@pytest.mark.gpu
@pytest.mark.parametrize("test,name", [(0, "qk_kmajor"), (1, "pv_mnmajor_ss"), (2, "pv_tmem_a")])
def test_tcgen05_block(test, name):
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.init()
    lib = _build()
    err = lib.fia_selftest_run(test)
    assert err >= 0, f"{name}: setup/timeout code {err}"
    assert err < 1e-3, f"{name}: max abs err {err}"
