"""GB300-native row-major FP32 GEMM (C = A x B) behind a small C ABI.

The kernels live in ``libtg_sgemm.so`` (built from ``csrc/`` for sm_103a);
``binding`` marshals torch tensors into the C ABI declared in
``include/tg_sgemm.h``.  ``workloads`` draws the seeded synthetic inputs.
"""
from .binding import (  # noqa: F401
    EXPORTS,
    PATHS,
    STATUS,
    TgError,
    error_site,
    host_blocks,
    host_device_bytes,
    lib,
    matmul,
    matmul_general,
    matmul_noalloc,
    plan,
    plan_general,
    selftest_wait_timeout,
    sgemm_host,
    status_string,
    reduce_plan,
    reduce_sum,
    sync_status,
    transpose,
)
