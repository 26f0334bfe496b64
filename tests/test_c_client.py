"""The boundary from plain C: tests/c/tg_c_client.c links libtg_sgemm.so
(and the oracle library) with gcc and calls the C ABI directly."""
import os
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "shared_memory_tiled_fp32_gb300")
ORACLE = os.path.join(ROOT, "oracle")


def build_client(tmp_path):
    import oracle
    import shared_memory_tiled_fp32_gb300 as tg

    tg.lib()
    oracle.load()
    exe = str(tmp_path / "tg_c_client")
    cuda_inc = "/usr/local/cuda/include"
    cmd = ["gcc", "-std=c11", "-O1", os.path.join(ROOT, "tests", "c", "tg_c_client.c"), "-o", exe,
           "-I", os.path.join(ROOT, "include"), "-I", cuda_inc,
           "-L", PKG, "-ltg_sgemm", "-L", ORACLE, "-ltg_oracle",
           f"-Wl,-rpath,{PKG}", f"-Wl,-rpath,{ORACLE}"]
    subprocess.run(cmd, check=True)
    return exe


def test_c_client_cpu_checks(tmp_path):
    r = subprocess.run([build_client(tmp_path), "cpu"], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and "C ABI OK" in r.stdout, r.stderr


@pytest.mark.gpu
def test_c_client_gpu_products(tmp_path):
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    r = subprocess.run([build_client(tmp_path), "gpu"], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and "C ABI OK" in r.stdout, r.stdout + r.stderr
