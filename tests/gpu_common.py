"""Shared helpers of the GPU parity tests: tolerance checks and cached oracle
references.  The references come only from the CPU oracle on the seeded
inputs of shared_memory_tiled_fp32_gb300.workloads."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from shared_memory_tiled_fp32_gb300.workloads import WORKLOADS, make_inputs, sample_rows

# Largest M*N*K whose every output the tests check (2^36 covers the 4096^3 and
# 2048 x 2048 x 16384 cases); above it, `row_sample` rows are checked.
FULL_CHECK_LIMIT = 2 ** 36

SENTINEL_BITS = 0x7FC0DEAD  # a quiet NaN no kernel produces


def assert_close(got: np.ndarray, ref: np.ndarray, K: int, what: str = ""):
    """The fp32 tolerance: normwise relative error <= 1e-5 and element-wise
    error <= 1e-4 * sqrt(K) * max|ref|, both over the checked set, in fp64."""
    g = got.astype(np.float64)
    r = ref.astype(np.float64)
    assert np.all(np.isfinite(g)), f"{what}: non-finite output"
    nr = np.linalg.norm(r)
    rel = np.linalg.norm(g - r) / nr if nr > 0 else np.linalg.norm(g)
    elt = np.abs(g - r).max() if g.size else 0.0
    bound = 1e-4 * np.sqrt(max(K, 1)) * (np.abs(r).max() if r.size else 0.0)
    assert rel <= 1e-5, f"{what}: normwise relative error {rel:.3e} > 1e-5"
    assert elt <= bound, f"{what}: element error {elt:.3e} > {bound:.3e}"
    return rel, elt


def assert_bitexact(got: np.ndarray, ref: np.ndarray, what: str = ""):
    """Bit equality with +0 and -0 counted equal."""
    g = (got.astype(np.float32) + np.float32(0.0)).view(np.uint32)
    r = (ref.astype(np.float32) + np.float32(0.0)).view(np.uint32)
    bad = np.argwhere(g != r)
    assert bad.size == 0, (f"{what}: {len(bad)} of {g.size} differ, first at {tuple(bad[0])}: "
                           f"{got[tuple(bad[0])]!r} vs {ref[tuple(bad[0])]!r}")


_refs: dict = {}


def workload_case(name: str):
    """(A, B, rows, ref) for a named workload; ref holds the oracle's rows
    `rows` (all rows when the whole product is checked).  Cached per session."""
    if name not in _refs:
        w = WORKLOADS[name]
        A, B = make_inputs(w.M, w.N, w.K, w.dist, w.seed)
        if w.M * w.N * w.K <= FULL_CHECK_LIMIT:
            rows = np.arange(w.M)
            ref = oracle.sgemm(A.numpy(), B.numpy())
        else:
            rows = sample_rows(w).numpy()
            ref = oracle.sgemm_rows(A.numpy(), B.numpy(), rows)
        _refs[name] = (A, B, rows, ref)
    return _refs[name]


def fill_sentinel(t: torch.Tensor):
    t.view(torch.int32).fill_(SENTINEL_BITS - (1 << 32) if SENTINEL_BITS >= 1 << 31 else SENTINEL_BITS)


def is_sentinel(x: np.ndarray) -> np.ndarray:
    return x.astype(np.float32).view(np.uint32) == SENTINEL_BITS
