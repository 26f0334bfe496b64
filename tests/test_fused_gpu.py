"""GPU parity of the 3xTF32 kernel's in-kernel split of A (raw A staged by
TMA, lo written beside it in shared memory) against the oracle.

The fused form is taken automatically for A stored M x K when its base and
row pitch are 16-byte aligned and the product runs on CTA pairs (B always
takes the pre-pass); TG_FUSED_SPLIT=0 turns it off.  Every case runs both
ways and both are checked against the oracle (bit for bit on integer
inputs), and the plan must report whether the kernel split A.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from gpu_common import assert_bitexact, assert_close
from shared_memory_tiled_fp32_gb300.workloads import make_inputs

pytestmark = pytest.mark.gpu


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


def general(tg, As, Bs, trans_a, trans_b, M, N, alpha=1.0, beta=0.0, C0=None, path="tf32x3", **kw):
    C = torch.zeros(M, N, device="cuda") if C0 is None else torch.from_numpy(C0.copy()).cuda()
    tg.matmul_general(torch.from_numpy(As).cuda(), torch.from_numpy(Bs).cuda(), C, trans_a=trans_a,
                      trans_b=trans_b, alpha=alpha, beta=beta, path=path, **kw)
    torch.cuda.synchronize()
    assert tg.sync_status() == 0
    return C.cpu().numpy()


def plan_flags(tg, As, Bs, trans_a, trans_b, M, N, K, path="tf32x3"):
    Ad, Bd = torch.from_numpy(As).cuda(), torch.from_numpy(Bs).cuda()
    C = torch.empty(M, N, device="cuda")
    p = tg.plan_general(trans_a, trans_b, M, N, K, Ad.stride(0), Bd.stride(0), C.stride(0), A=Ad.data_ptr(),
                        B=Bd.data_ptr(), C=C.data_ptr(), path=path)
    return p["fused_split"]


SHAPES = [(129, 300, 700), (256, 256, 16), (300, 513, 17), (383, 257, 4097), (1000, 3000, 1100),
          (640, 256, 2048), (2048, 2048, 4096)]


@pytest.mark.parametrize("path", ["tf32x3", "tf32bf16"])
@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("trans_a,trans_b", [(False, False), (False, True), (True, True)])
def test_fused_split_matches_oracle(tg, M, N, K, trans_a, trans_b, path, monkeypatch):
    A, B = (x.numpy() for x in make_inputs(M, N, K, "uniform", 1300 + M + K))
    As, Bs = stored(A, trans_a), stored(B, trans_b)
    ref = oracle.sgemm(A, B)
    # raw A: stored M x K with a 16-byte row pitch (lda = K here)
    want = 1 if K % 4 == 0 and not trans_a else 0
    for fused in ("1", "0"):
        monkeypatch.setenv("TG_FUSED_SPLIT", fused)
        assert plan_flags(tg, As, Bs, trans_a, trans_b, M, N, K, path) == (want if fused == "1" else 0)
        for split in (0, 1, 3):
            got = general(tg, As, Bs, trans_a, trans_b, M, N, split_k=split, path=path)
            assert_close(got, ref, K, f"{path} fused={fused} op=({trans_a},{trans_b}) {M}x{N}x{K} s{split}")


@pytest.mark.parametrize("path", ["tf32x3", "tf32bf16"])
@pytest.mark.parametrize("trans_b", [False, True])
def test_fused_split_integers_bitexact(tg, trans_b, path):
    """Integer data: the raw value is its own hi (lo = 0), so the products are
    exact, on every split and tail form."""
    for i, (M, N, K) in enumerate([(129, 300, 700), (1000, 3000, 1100), (2048, 2048, 2049), (300, 513, 17)]):
        A, B = (x.numpy() for x in make_inputs(M, N, K, "int", 1400 + i))
        ref = oracle.sgemm(A, B)
        for split in (0, 2):
            got = general(tg, A, stored(B, trans_b), False, trans_b, M, N, split_k=split, path=path)
            assert_bitexact(got, ref, f"{path} integers trans_b={trans_b} {M}x{N}x{K} s{split}")


def test_fused_split_strided_and_scaled(tg):
    """A row pitch larger than K (still 16-byte aligned: the raw copy reads
    only the first K columns; the rest must not leak in), alpha/beta."""
    M, N, K, lda = 777, 1029, 513, 520
    A, B = (x.numpy() for x in make_inputs(M, N, K, "uniform", 1500))
    Abuf = np.full((M, lda), np.nan, np.float32)  # padding columns: NaN would poison the result
    Abuf[:, :K] = A
    Ad = torch.from_numpy(Abuf).cuda()[:, :K]
    Bd = torch.from_numpy(B).cuda()
    C0 = np.random.default_rng(3).uniform(-1, 1, (M, N)).astype(np.float32)
    C = torch.from_numpy(C0.copy()).cuda()
    p = tg.plan_general(False, False, M, N, K, lda, N, N, A=Ad.data_ptr(), B=Bd.data_ptr(), C=C.data_ptr(),
                        path="tf32x3")
    assert p["fused_split"] == 1
    tg.matmul_general(Ad, Bd, C, alpha=0.5, beta=1.0, path="tf32x3")
    torch.cuda.synchronize()
    assert tg.sync_status() == 0
    ref = oracle.sgemm_general(0, 0, 0.5, A, B, 1.0, C0.copy())
    assert_close(C.cpu().numpy(), ref, K, "strided A, alpha/beta")


def test_fused_split_unaligned_falls_back(tg):
    """A sub-view starting 4 bytes into its buffer is not TMA-legal: the
    pre-pass splits it, with the same result."""
    M, N, K = 300, 260, 96
    A, B = (x.numpy() for x in make_inputs(M, N, K, "uniform", 1600))
    buf = torch.zeros(1 + M * K, device="cuda")
    Av = buf[1:].view(M, K)
    Av.copy_(torch.from_numpy(A).cuda())
    Bd = torch.from_numpy(B).cuda()
    C = torch.empty(M, N, device="cuda")
    p = tg.plan(M, N, K, A=Av.data_ptr(), B=Bd.data_ptr(), C=C.data_ptr(), path="tf32x3")
    assert p["fused_split"] == 0
    tg.matmul(Av, Bd, out=C, path="tf32x3")
    torch.cuda.synchronize()
    assert_close(C.cpu().numpy(), oracle.sgemm(A, B), K, "unaligned A")


def test_fused_split_special_values(tg):
    """A NaN in row i of A makes row i of C NaN; operands near the largest
    float stay finite (truncating to tf32 never overflows)."""
    M, N, K = 260, 300, 64
    A, B = (x.numpy() for x in make_inputs(M, N, K, "uniform", 1700))
    A[5, 17] = np.nan
    got = general(tg, A, B, False, False, M, N)
    assert np.all(np.isnan(got[5]))
    mask = np.ones(M, bool)
    mask[5] = False
    ref = oracle.sgemm(A, B)
    assert_close(got[mask], ref[mask], K, "rows without NaN")
    fmax = np.finfo(np.float32).max
    big = (np.random.default_rng(9).uniform(0.9996, 1.0, (M, K)) * fmax).astype(np.float32)
    small = (np.random.default_rng(10).uniform(-1, 1, (K, N)) * 2.0 ** -100).astype(np.float32)
    got = general(tg, big, small, False, False, M, N)
    assert np.all(np.isfinite(got))
    assert_close(got, oracle.sgemm(big, small), K, "near FLT_MAX")
