"""Seeded random configurations of tg_sgemm_general against the oracle:
shapes (including tile edges and sizes past one round of CTAs), leading
dimensions, unaligned sub-view offsets, op forms, alpha/beta, both math paths,
and automatic or explicit K splits.  Each case also checks that nothing
outside the output block changes."""
import numpy as np
import pytest
import torch

import oracle
from gpu_common import assert_close, fill_sentinel, is_sentinel

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tg():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import shared_memory_tiled_fp32_gb300 as tg

    torch.cuda.set_device(0)
    tg.lib()
    return tg


def draw_case(rng):
    edges = [1, 3, 31, 127, 128, 129, 255, 256, 257, 513]
    pick = lambda: int(rng.choice(edges)) if rng.random() < 0.4 else int(rng.integers(1, 1100))
    M, N, K = pick(), pick(), pick()
    if rng.random() < 0.15:  # sometimes large enough for pairs and last-round balancing
        M, N = int(rng.integers(2000, 4200)), int(rng.integers(600, 2100))
    op_a, op_b = int(rng.integers(0, 2)), int(rng.integers(0, 2))
    alpha = float(rng.choice([1.0, 1.0, -0.5, 2.0, 0.3]))
    beta = float(rng.choice([0.0, 0.0, 1.0, -1.5]))
    path = str(rng.choice(["tf32x3", "ffma", "tiled"]))
    split = int(rng.choice([0, 0, 1, 2, 5]))
    pads = [int(rng.integers(0, 6)) for _ in range(3)]
    offs = [int(rng.integers(0, 4)) for _ in range(3)]
    return M, N, K, op_a, op_b, alpha, beta, path, split, pads, offs


def strided(dev_rows, dev_cols, pad, off, host):
    """A device view of `host` with row pitch cols + pad, starting `off`
    floats into its buffer (so it may be unaligned)."""
    ld = dev_cols + pad
    buf = torch.zeros(off + dev_rows * ld + 1, device="cuda")
    view = buf[off:off + dev_rows * ld].view(dev_rows, ld)[:, :dev_cols]
    view.copy_(torch.from_numpy(host))
    return view


@pytest.mark.parametrize("seed", range(32))
def test_fuzz_general(tg, seed):
    rng = np.random.default_rng(1000 + seed)
    M, N, K, op_a, op_b, alpha, beta, path, split, pads, offs = draw_case(rng)
    if seed >= 24:  # the opt-in tf32 + bf16 cross-product path
        path = "tf32bf16"
    A = rng.uniform(-1, 1, (M, K)).astype(np.float32)
    B = rng.uniform(-1, 1, (K, N)).astype(np.float32)
    C0 = rng.uniform(-1, 1, (M, N)).astype(np.float32)
    As = np.ascontiguousarray(A.T) if op_a else A
    Bs = np.ascontiguousarray(B.T) if op_b else B
    Ad = strided(As.shape[0], As.shape[1], pads[0], offs[0], As)
    Bd = strided(Bs.shape[0], Bs.shape[1], pads[1], offs[1], Bs)
    ldc, guard = N + pads[2], 256
    cbuf = torch.empty(2 * guard + offs[2] + M * ldc, device="cuda")
    fill_sentinel(cbuf)
    base = guard + offs[2]
    Cd = cbuf[base:base + M * ldc].view(M, ldc)[:, :N]
    Cd.copy_(torch.from_numpy(C0))
    tg.matmul_general(Ad, Bd, Cd, trans_a=bool(op_a), trans_b=bool(op_b), alpha=alpha, beta=beta, path=path,
                      split_k=split)
    torch.cuda.synchronize()
    assert tg.sync_status() == 0
    host = cbuf.cpu().numpy()
    idx = base + (np.arange(M)[:, None] * ldc + np.arange(N)[None, :])
    inside = np.zeros(host.shape, bool)
    inside[idx.ravel()] = True
    assert np.all(is_sentinel(host[~inside])), f"case {seed}: write outside C"
    if M * N * K <= 2e8:
        ref = oracle.sgemm_general(op_a, op_b, alpha, As, Bs, beta, C0.copy())
    else:  # the plain oracle on op(A), op(B) (the same bits as the general form), scaled in double
        prod = oracle.sgemm(A, B).astype(np.float64)
        ref = (alpha * prod + (beta * C0.astype(np.float64) if beta != 0.0 else 0.0)).astype(np.float32)
    what = f"case {seed}: {M}x{N}x{K} op=({op_a},{op_b}) a={alpha} b={beta} {path} s={split} pads={pads} offs={offs}"
    assert_close(host[idx], ref, K, what)
