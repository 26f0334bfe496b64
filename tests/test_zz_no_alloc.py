"""tg_sgemm_noalloc: the product for callers that cannot allocate device
memory at call time (its scratch is a fixed device array the library holds).

Called through the C ABI with ctypes and compared, within the tolerance of
the other parity tests, with the output of the allocating entry point
tg_sgemm_ex on the same inputs, for two calls in a row with different
inputs (the second call runs on scratch left over from the first).  This file
is collected last on purpose; it also runs on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

from gpu_common import assert_close
from shared_memory_tiled_fp32_gb300.workloads import make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import shared_memory_tiled_fp32_gb300 as tg

    torch.cuda.set_device(0)
    return tg.lib()


def _noalloc(L, A, B, C, stream):
    M, K = A.shape
    N = B.shape[1]
    return L.tg_sgemm_noalloc(M, N, K, A.data_ptr(), A.stride(0), B.data_ptr(), B.stride(0),
                              C.data_ptr(), C.stride(0), ctypes.c_void_p(stream.cuda_stream))


@pytest.mark.parametrize("M,N,K", [(777, 1029, 513), (1024, 1024, 1024), (130, 300, 2000)])
def test_noalloc_matches_allocating_entry(lib, M, N, K):
    import shared_memory_tiled_fp32_gb300 as tg

    stream = torch.cuda.current_stream()
    for call, seed in enumerate((31, 32)):  # two calls in a row, different inputs
        A, B = make_inputs(M, N, K, "uniform", seed + M)
        Ad, Bd = A.cuda(), B.cuda()
        C_ref = tg.matmul(Ad, Bd, path="tf32x3")
        C = torch.full((M, N), float("nan"), device="cuda")
        assert _noalloc(lib, Ad, Bd, C, stream) == 0
        torch.cuda.synchronize()
        assert tg.sync_status() == 0
        assert_close(C.cpu().numpy(), C_ref.cpu().numpy(), K, f"noalloc call {call} {M}x{N}x{K}")


def test_noalloc_rejects_oversized_products(lib):
    limit = 64 << 20
    M, N = 512, 8192
    K = 2048  # B's hi/lo copies alone: 8 * N * K = 128 MiB > 64 MiB
    assert 8 * N * K > limit
    A = torch.empty(M, K, device="cuda")
    B = torch.empty(K, N, device="cuda")
    C = torch.empty(M, N, device="cuda")
    assert _noalloc(lib, A, B, C, torch.cuda.current_stream()) == 6  # TG_ERR_WORKSPACE_TOO_SMALL
