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


def _scratch_bytes(M, N, K, a_in_kernel):
    """The hi/lo split tiles: rows padded to whole 256-row tile pairs (128 for
    a single tile row), K to a multiple of 16, 8 bytes per element; none for
    A when the GEMM kernel splits it itself (A's base and row pitch 16-byte
    aligned, more than one 128-row tile)."""
    rup = lambda x, m: -(-x // m) * m
    a_rows = 0 if a_in_kernel else (rup(M, 256) if M > 128 else 128)
    return 8 * (a_rows + rup(N, 256)) * rup(K, 16)


def _a_in_kernel(M, K, fused):
    return fused and M > 128 and K % 4 == 0


# At the 64 MiB limit exactly (the planner's balanced-tail partials then do
# not fit, so the call re-plans without them): 2048^3 with A split by the
# pre-pass, 2048 x 4096 x 2048 with A split in the kernel.
@pytest.mark.parametrize("fused", [True, False])
@pytest.mark.parametrize("M,N,K", [(777, 1029, 513), (1024, 1024, 1024), (130, 300, 2000), (2048, 2048, 2048),
                                   (2048, 4096, 2048)])
def test_noalloc_matches_allocating_entry_and_oracle(lib, M, N, K, fused, monkeypatch):
    import shared_memory_tiled_fp32_gb300 as tg

    monkeypatch.setenv("TG_FUSED_SPLIT", "1" if fused else "0")
    need = _scratch_bytes(M, N, K, _a_in_kernel(M, K, fused))
    if need > LIMIT:
        pytest.skip("does not fit this form's scratch (the rejection test covers it)")
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


@pytest.mark.parametrize("fused", [True, False])
def test_noalloc_rejects_oversized_products(lib, fused, monkeypatch):
    monkeypatch.setenv("TG_FUSED_SPLIT", "1" if fused else "0")
    stream = torch.cuda.current_stream()
    cases = [(512, 8192, 2048), (2048, 4097, 2048), (2048, 4096, 2049), (128, 4097, 2048)]
    if not fused:
        cases += [(2048, 2049, 2048), (2048, 2048, 2049)]
    for M, N, K in cases:
        assert _scratch_bytes(M, N, K, _a_in_kernel(M, K, fused)) > LIMIT, (M, N, K)
        A = torch.empty(M, K, device="cuda")
        B = torch.empty(K, N, device="cuda")
        C = torch.empty(M, N, device="cuda")
        assert _noalloc(lib, A, B, C, stream) == TOO_SMALL, (M, N, K)
