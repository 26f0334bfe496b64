"""GPU parity of tg_transpose (all four variants) against the oracle's index
permutation: bit-exact, with sentinel bands around the output."""
import numpy as np
import pytest
import torch

import oracle
from gpu_common import fill_sentinel, is_sentinel

pytestmark = pytest.mark.gpu

VARIANTS = ["direct", "tile32", "padded", "swizzled"]


@pytest.fixture(scope="module")
def tg():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import shared_memory_tiled_fp32_gb300 as tg

    torch.cuda.set_device(0)
    tg.lib()
    return tg


@pytest.mark.parametrize("variant", VARIANTS)
def test_transpose_shapes(tg, variant):
    rng = np.random.default_rng(3)
    for (r, c) in [(1, 1), (1, 33), (31, 1), (32, 32), (33, 31), (1000, 777), (4097, 1025)]:
        X = rng.standard_normal((r, c)).astype(np.float32)
        got = tg.transpose(torch.from_numpy(X).cuda(), variant=variant)
        torch.cuda.synchronize()
        assert np.array_equal(got.cpu().numpy().view(np.uint32), oracle.transpose(X).view(np.uint32)), (variant, r, c)


@pytest.mark.parametrize("variant", VARIANTS)
def test_transpose_full_size(tg, variant):
    """8192 x 8192 (256 MiB, larger than L2) and 16384 x 1024: every block of
    the one-wave grid runs many iterations of its grid-stride loop, as in the
    benchmarked 16384^2 case; the whole output is compared bit for bit."""
    for i, (r, c) in enumerate([(8192, 8192), (16384, 1024)]):
        X = np.random.default_rng(40 + i).standard_normal((r, c)).astype(np.float32)
        got = tg.transpose(torch.from_numpy(X).cuda(), variant=variant)
        torch.cuda.synchronize()
        assert np.array_equal(got.cpu().numpy().view(np.uint32), oracle.transpose(X).view(np.uint32)), (variant, r, c)


@pytest.mark.parametrize("variant", VARIANTS)
def test_transpose_strided_with_canaries(tg, variant):
    rows, cols, ld_in, ld_out, guard = 70, 45, 53, 77, 512
    X = np.random.default_rng(4).uniform(-1, 1, (rows, ld_in)).astype(np.float32)
    Xd = torch.from_numpy(X).cuda()[:, :cols]
    buf = torch.empty(2 * guard + cols * ld_out, device="cuda")
    fill_sentinel(buf)
    out = buf[guard:guard + cols * ld_out].view(cols, ld_out)[:, :rows]
    tg.transpose(Xd, out, variant=variant)
    torch.cuda.synchronize()
    host = buf.cpu().numpy()
    idx = guard + (np.arange(cols)[:, None] * ld_out + np.arange(rows)[None, :])
    inside = np.zeros(host.shape, bool)
    inside[idx.ravel()] = True
    assert np.all(is_sentinel(host[~inside])), "write outside the output block"
    assert np.array_equal(host[idx].view(np.uint32), oracle.transpose(X[:, :cols]).view(np.uint32))


def test_transpose_rejects_bad_arguments(tg):
    import ctypes

    L = tg.lib()
    x = torch.empty(8, 8, device="cuda")
    y = torch.empty(8, 8, device="cuda")
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert L.tg_transpose(7, 8, 8, x.data_ptr(), 8, y.data_ptr(), 8, s) == 1     # bad variant
    assert L.tg_transpose(1, 8, 8, x.data_ptr(), 7, y.data_ptr(), 8, s) == 1     # ld_in < cols
    assert L.tg_transpose(1, 8, 8, x.data_ptr(), 8, x.data_ptr(), 8, s) == 1     # in place
    assert L.tg_transpose(1, 0, 8, x.data_ptr(), 8, y.data_ptr(), 1, s) == 0     # empty
