"""GPU parity of tg_reduce_sum (all five variants) against the oracle's
double-accumulated sum.  Bound: an fp32 summation whose longest chain of
additions from an input to the result has d steps is within d * 2^-24 *
sum|x| of the exact sum; d is taken per variant from its structure.  Integer
inputs with partial sums below 2^24 are exact on every variant."""
import math

import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu

VARIANTS = ["interleaved", "sequential", "shuffle", "atomic", "fast"]


@pytest.fixture(scope="module")
def tg():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import shared_memory_tiled_fp32_gb300 as tg

    torch.cuda.set_device(0)
    tg.lib()
    return tg


def chain_bound(variant, n, sms):
    lg = max(1, math.ceil(math.log2(max(n, 2))))
    if variant == "atomic":
        return 8 + math.ceil(n / 256)          # block tree + one atomic add per block, any order
    if variant == "fast":
        threads = 4 * sms * 256
        return math.ceil(n / (4 * threads)) + 16 + math.ceil(4 * sms / 256) + 16
    return lg + 8


@pytest.mark.parametrize("variant", VARIANTS)
def test_reduce_against_oracle(tg, variant):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    rng = np.random.default_rng(13)
    for n in (1, 2, 255, 256, 257, 1000, 65536 + 3, 2 ** 20 + 17, 2 ** 24):
        x = rng.standard_normal(n).astype(np.float32)
        xd = torch.from_numpy(x).cuda()
        for off in (0, 1):  # an unaligned start exercises the head path of the float4 loop
            xs = xd[off:] if n > 1 else xd
            got = float(tg.reduce_sum(xs, variant=variant).item())
            ref = float(oracle.reduce_sum(x[off:] if n > 1 else x))
            bound = chain_bound(variant, xs.numel(), sms) * 2.0 ** -24 * float(np.abs(x).sum())
            assert abs(got - ref) <= bound, (variant, n, off, got, ref, bound)


@pytest.mark.parametrize("variant", VARIANTS)
def test_reduce_integer_exact_and_empty(tg, variant):
    rng = np.random.default_rng(14)
    x = rng.integers(-2, 3, 3 * 2 ** 20 + 5).astype(np.float32)
    got = tg.reduce_sum(torch.from_numpy(x).cuda(), variant=variant).item()
    assert got == float(oracle.reduce_sum(x)) == float(x.astype(np.int64).sum())
    z = tg.reduce_sum(torch.empty(0, device="cuda"), variant=variant).item()
    assert z == 0.0


@pytest.mark.parametrize("variant", ["interleaved", "sequential", "shuffle", "fast"])
def test_reduce_deterministic(tg, variant):
    x = torch.from_numpy(np.random.default_rng(15).standard_normal(2 ** 22).astype(np.float32)).cuda()
    a = tg.reduce_sum(x, variant=variant).cpu().numpy().view(np.uint32)
    b = tg.reduce_sum(x, variant=variant).cpu().numpy().view(np.uint32)
    assert np.array_equal(a, b)
