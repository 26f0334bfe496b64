"""GPU parity of tg_sgemm_general: C = alpha * op(A) op(B) + beta * C with
stored-transposed operands (the forward/backward products of a fully
connected layer), against the oracle's general form.  Tolerances as in
test_gemm_gpu.py; bit-exact on integer data with integer alpha/beta."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from gpu_common import assert_bitexact, assert_close
from shared_memory_tiled_fp32_gb300.workloads import make_inputs

pytestmark = pytest.mark.gpu

OPS = [(0, 0), (1, 0), (0, 1), (1, 1)]


@pytest.fixture(scope="module")
def tg():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import shared_memory_tiled_fp32_gb300 as tg

    tg.lib()
    torch.cuda.set_device(0)
    return tg


def stored(X, trans):
    return np.ascontiguousarray(X.T) if trans else np.ascontiguousarray(X)


def gpu_general(tg, op_a, op_b, alpha, As, Bs, beta, C0, **kw):
    C = torch.from_numpy(C0.copy()).cuda()
    tg.matmul_general(torch.from_numpy(As).cuda(), torch.from_numpy(Bs).cuda(), C, trans_a=bool(op_a),
                      trans_b=bool(op_b), alpha=alpha, beta=beta, **kw)
    torch.cuda.synchronize()
    assert tg.sync_status() == 0
    return C.cpu().numpy()


@pytest.mark.parametrize("path", ["tf32x3", "ffma", "tiled", "tf32bf16"])
@pytest.mark.parametrize("op_a,op_b", OPS)
def test_general_ops_alpha_beta(tg, path, op_a, op_b):
    M, N, K = 300, 257, 513
    A, B = make_inputs(M, N, K, "uniform", 70 + 2 * op_a + op_b)
    A, B = A.numpy(), B.numpy()
    As, Bs = stored(A, op_a), stored(B, op_b)
    C0 = np.random.default_rng(5).uniform(-1, 1, (M, N)).astype(np.float32)
    for alpha, beta in [(1.0, 0.0), (2.5, -0.75), (-1.0, 1.0)]:
        ref = oracle.sgemm_general(op_a, op_b, alpha, As, Bs, beta, C0.copy())
        for split in (0, 1, 3):
            got = gpu_general(tg, op_a, op_b, alpha, As, Bs, beta, C0, path=path, split_k=split)
            assert_close(got, ref, K, f"{path} op=({op_a},{op_b}) a={alpha} b={beta} s={split}")


@pytest.mark.parametrize("path", ["tf32x3", "ffma", "tiled", "tf32bf16"])
@pytest.mark.parametrize("op_a,op_b", OPS)
def test_general_integer_bitexact(tg, path, op_a, op_b):
    M, N, K = 130, 270, 300
    A, B = make_inputs(M, N, K, "int", 80 + 2 * op_a + op_b)
    A, B = A.numpy(), B.numpy()
    As, Bs = stored(A, op_a), stored(B, op_b)
    C0 = np.random.default_rng(6).integers(-9, 10, (M, N)).astype(np.float32)
    ref = oracle.sgemm_general(op_a, op_b, 2.0, As, Bs, -1.0, C0.copy())
    for split in (0, 2):
        assert_bitexact(gpu_general(tg, op_a, op_b, 2.0, As, Bs, -1.0, C0, path=path, split_k=split), ref,
                        f"{path} op=({op_a},{op_b}) s={split}")


@pytest.mark.parametrize("path", ["tf32x3", "ffma"])
def test_general_ragged_alpha_beta(tg, path):
    """The ragged workload shape (777 x 1029 x 513: no dimension a tile
    multiple, ldc = 1029 so C rows are not 16-byte aligned) with alpha = 0.5
    and beta = 1: exercises the scaled epilogue's partial row blocks (fewer
    than 32 rows, columns past N) on both GEMM kernels, with and without a
    split of K and with the planner's own choice."""
    M, N, K = 777, 1029, 513
    A, B = make_inputs(M, N, K, "uniform", 3)
    A, B = A.numpy(), B.numpy()
    C0 = np.random.default_rng(11).uniform(-1, 1, (M, N)).astype(np.float32)
    ref = oracle.sgemm_general(0, 0, 0.5, A, B, 1.0, C0.copy())
    for split in (0, 1, 2):
        got = gpu_general(tg, 0, 0, 0.5, A, B, 1.0, C0, path=path, split_k=split)
        assert_close(got, ref, K, f"{path} ragged alpha=0.5 beta=1 s={split}")
    Ai, Bi = (x.numpy() for x in make_inputs(M, N, K, "int", 12))
    Ci = np.random.default_rng(13).integers(-9, 10, (M, N)).astype(np.float32)
    assert_bitexact(gpu_general(tg, 0, 0, 0.5, Ai, Bi, 1.0, Ci, path=path),
                    oracle.sgemm_general(0, 0, 0.5, Ai, Bi, 1.0, Ci.copy()), f"{path} ragged integers")


def test_general_k0_and_beta0_ignores_c(tg):
    M, N = 9, 11
    C0 = np.random.default_rng(7).uniform(-1, 1, (M, N)).astype(np.float32)
    for path in ("tf32x3", "ffma", "tiled", "tf32bf16"):
        got = gpu_general(tg, 1, 1, 3.0, np.zeros((0, M), np.float32), np.zeros((N, 0), np.float32), 0.5, C0,
                          path=path)
        assert_bitexact(got, 0.5 * C0, f"K=0 {path}")
        A, B = make_inputs(M, N, 40, "uniform", 8)
        nan_c = np.full((M, N), np.nan, np.float32)
        got = gpu_general(tg, 0, 0, 1.5, A.numpy(), B.numpy(), 0.0, nan_c, path=path)
        assert np.all(np.isfinite(got)), f"beta=0 read C on {path}"
        assert_close(got, oracle.sgemm_general(0, 0, 1.5, A.numpy(), B.numpy(), 0.0, nan_c.copy()), 40, path)


@pytest.mark.parametrize("op_a,op_b", [(1, 0), (0, 1)])
def test_general_large_backward_shapes(tg, op_a, op_b):
    """dW = X^T dY (A stored transposed) and dX = dY W^T (B stored
    transposed) at 2048 x 2048 x 4096 with the planner's choices (CTA pairs,
    last-round balancing), alpha = 0.5, beta = 1, checked on 256 sampled rows
    against the oracle applied to explicitly transposed copies."""
    M, N, K = 2048, 2048, 4096
    A, B = make_inputs(M, N, K, "normal", 90 + op_a)
    A, B = A.numpy(), B.numpy()
    As, Bs = stored(A, op_a), stored(B, op_b)
    C0 = np.random.default_rng(9).standard_normal((M, N)).astype(np.float32)
    got = gpu_general(tg, op_a, op_b, 0.5, As, Bs, 1.0, C0)
    rows = np.sort(np.random.default_rng(10).choice(M, 256, replace=False))
    prod = oracle.sgemm_rows(A, B, rows).astype(np.float64)  # op(A) op(B) rows, pinned oracle
    ref = (0.5 * prod + 1.0 * C0[rows].astype(np.float64)).astype(np.float32)
    assert_close(got[rows], ref, K, f"backward op=({op_a},{op_b})")
