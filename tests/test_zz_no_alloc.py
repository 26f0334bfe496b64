"""tg_sgemm_noalloc: the product for callers that cannot allocate device
memory at call time (its scratch is a fixed device array the library holds).

Called through the C ABI with ctypes.  Each case makes two calls in a row
with different inputs, so the second call runs on scratch left over from the
first; every call is compared with the allocating entry point's output on the
same inputs (within the tolerance of the other parity tests) and with the CPU
oracle (the same tolerance; bit for bit on integer inputs, which shows that
no stale scratch bits reach the result).  This file is collected last on
purpose; it also runs on its own in a fresh process.
"""
import ctypes

import pytest
import torch

import oracle
from gpu_common import assert_bitexact, assert_close
from shared_memory_tiled_fp32_gb300.workloads import make_inputs

pytestmark = pytest.mark.gpu

LIMIT = 64 << 20  # TG_SGEMM_NOALLOC_SCRATCH_BYTES
TOO_SMALL = 6     # TG_ERR_WORKSPACE_TOO_SMALL


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


def _scratch_bytes(M, N, K):
    """The hi/lo split tiles: rows padded to whole 256-row tile pairs (128 for
    a single tile row), K to a multiple of 16, 8 bytes per element."""
    rup = lambda x, m: -(-x // m) * m
    return 8 * ((rup(M, 256) if M > 128 else 128) + rup(N, 256)) * rup(K, 16)


# (2048, 2048, 2048): the split tiles fill the 64 MiB exactly, so the
# planner's balanced-tail partials do not fit and the call re-plans without them
@pytest.mark.parametrize("M,N,K", [(777, 1029, 513), (1024, 1024, 1024), (130, 300, 2000), (2048, 2048, 2048)])
def test_noalloc_matches_allocating_entry_and_oracle(lib, M, N, K):
    import shared_memory_tiled_fp32_gb300 as tg

    assert _scratch_bytes(M, N, K) <= LIMIT
    stream = torch.cuda.current_stream()
    for call, (dist, seed) in enumerate((("uniform", 31), ("int", 32))):  # two calls in a row
        A, B = make_inputs(M, N, K, dist, seed + M)
        Ad, Bd = A.cuda(), B.cuda()
        C_ref = tg.matmul(Ad, Bd, path="tf32x3")
        C = torch.full((M, N), float("nan"), device="cuda")
        assert _noalloc(lib, Ad, Bd, C, stream) == 0
        torch.cuda.synchronize()
        assert tg.sync_status() == 0
        got = C.cpu().numpy()
        what = f"noalloc call {call} {M}x{N}x{K} {dist}"
        assert_close(got, C_ref.cpu().numpy(), K, what + " vs tg_sgemm")
        ref = oracle.sgemm(A.numpy(), B.numpy())
        if dist == "int":
            assert_bitexact(got, ref, what + " vs oracle")
        else:
            assert_close(got, ref, K, what + " vs oracle")


def test_noalloc_rejects_oversized_products(lib):
    stream = torch.cuda.current_stream()
    for M, N, K in [(512, 8192, 2048), (2048, 2049, 2048), (2048, 2048, 2049)]:
        assert _scratch_bytes(M, N, K) > LIMIT
        A = torch.empty(M, K, device="cuda")
        B = torch.empty(K, N, device="cuda")
        C = torch.empty(M, N, device="cuda")
        assert _noalloc(lib, A, B, C, stream) == TOO_SMALL, (M, N, K)
