"""Failure detection without a GPU fault: a kernel waits on an mbarrier that
nothing arrives on; its bounded wait gives up after a short limit, records a
timeout in the device error word and returns.  The host reads TG_ERR_TIMEOUT,
and the context stays usable for the next product."""
import numpy as np
import pytest
import torch

import oracle
from gpu_common import assert_close
from shared_memory_tiled_fp32_gb300.workloads import make_inputs

pytestmark = pytest.mark.gpu


def test_wait_gives_up_and_context_survives():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import shared_memory_tiled_fp32_gb300 as tg

    torch.cuda.set_device(0)
    assert tg.sync_status() == 0
    assert tg.selftest_wait_timeout(50_000) == 0  # 50 ms limit
    assert tg.error_site() == 0x301
    assert tg.sync_status() == 5  # TG_ERR_TIMEOUT, and the word is cleared
    assert tg.sync_status() == 0
    A, B = make_inputs(100, 120, 140, "uniform", 77)
    C = tg.matmul(A.cuda(), B.cuda())
    torch.cuda.synchronize()
    assert tg.sync_status() == 0
    assert_close(C.cpu().numpy(), oracle.sgemm(A.numpy(), B.numpy()), 140, "after timeout")


def test_selftest_rejects_bad_limits():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import shared_memory_tiled_fp32_gb300 as tg

    assert tg.selftest_wait_timeout(0) == 1
    assert tg.selftest_wait_timeout(20_000_000) == 1
