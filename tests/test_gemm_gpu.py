"""GPU parity of the C-ABI FP32 GEMM against the CPU oracle.

Every call goes through the C ABI (ctypes binding of libtg_sgemm.so).  Inputs
are the seeded synthetic workloads; references come from the oracle only.
Tolerances: bit-exact on integer-valued inputs (partial sums exact in fp32);
otherwise normwise relative error <= 1e-5 and element-wise error
<= 1e-4 * sqrt(K) * max|ref| (gpu_common.assert_close).
"""
from __future__ import annotations

import os

import numpy as np
import pytest
import torch

import oracle
from gpu_common import (assert_bitexact, assert_close, fill_sentinel, is_sentinel,
                        workload_case)
from shared_memory_tiled_fp32_gb300.workloads import WORKLOADS, make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tg():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import shared_memory_tiled_fp32_gb300 as tg

    tg.lib()  # must load: no fallback exists
    torch.cuda.set_device(0)
    return tg


def run(tg, A, B, **kw):
    C = tg.matmul(A.cuda(), B.cuda(), **kw)
    torch.cuda.synchronize()
    assert tg.sync_status() == 0
    return C.cpu().numpy()


# (workload, path, split_k) -- split_k 0 = the planner's choice, which is also
# what the headline bench runs
CASES = [
    ("sq256_uniform", "tf32x3", 0), ("sq256_uniform", "tf32x3", 1), ("sq256_uniform", "tf32x3", 5),
    ("sq256_uniform", "ffma", 0), ("sq256_uniform", "ffma", 1),
    ("sq256_int", "tf32x3", 0), ("sq256_int", "tf32x3", 1), ("sq256_int", "ffma", 0),
    ("ragged_777x1029x513", "tf32x3", 0), ("ragged_777x1029x513", "tf32x3", 1),
    ("ragged_777x1029x513", "tf32x3", 3), ("ragged_777x1029x513", "ffma", 0),
    ("ragged_777x1029x513", "ffma", 1),
    ("sq4096_uniform", "tf32x3", 0), ("sq4096_uniform", "tf32x3", 1), ("sq4096_uniform", "ffma", 0),
    ("sq4096_int", "tf32x3", 0), ("sq4096_int", "ffma", 0),
    ("sq8192_normal", "tf32x3", 0), ("sq8192_normal", "ffma", 0),
    ("longk_2048x2048x16384_normal", "tf32x3", 0), ("longk_2048x2048x16384_normal", "tf32x3", 2),
    ("longk_2048x2048x16384_normal", "tf32x3", 4), ("longk_2048x2048x16384_normal", "ffma", 0),
    ("sq256_uniform", "tiled", 0), ("sq256_int", "tiled", 0), ("ragged_777x1029x513", "tiled", 0),
    ("sq4096_int", "tiled", 0), ("sq4096_uniform", "auto", 0), ("sq256_uniform", "auto", 0),
    ("sq256_uniform", "tf32bf16", 0), ("sq256_int", "tf32bf16", 0), ("sq256_int", "tf32bf16", 1),
    ("ragged_777x1029x513", "tf32bf16", 0), ("ragged_777x1029x513", "tf32bf16", 3),
    ("sq4096_uniform", "tf32bf16", 0), ("sq4096_int", "tf32bf16", 0), ("sq8192_normal", "tf32bf16", 0),
    ("longk_2048x2048x16384_normal", "tf32bf16", 0), ("longk_2048x2048x16384_normal", "tf32bf16", 4),
]


@pytest.mark.parametrize("name,path,split", CASES, ids=[f"{n}-{p}-s{s}" for n, p, s in CASES])
def test_workload(tg, name, path, split):
    w = WORKLOADS[name]
    A, B, rows, ref = workload_case(name)
    C = run(tg, A, B, path=path, split_k=split)
    got = C[rows]
    if w.dist == "int":
        assert_bitexact(got, ref, f"{name} {path} split {split}")
    else:
        assert_close(got, ref, w.K, f"{name} {path} split {split}")


@pytest.mark.parametrize("path", ["tf32x3", "ffma", "tiled", "tf32bf16"])
def test_ragged_random_shapes(tg, path):
    """Shapes around tile edges and random shapes in [1, 300]^3."""
    rng = np.random.default_rng(7)
    shapes = [(1, 1, 1), (1, 257, 1), (129, 1, 33), (127, 255, 15), (128, 256, 16),
              (129, 257, 17), (128, 256, 32), (129, 257, 33), (3, 5, 1000)]
    shapes += [tuple(int(v) for v in rng.integers(1, 301, size=3)) for _ in range(10)]
    for i, (M, N, K) in enumerate(shapes):
        A, B = make_inputs(M, N, K, "uniform", 500 + i)
        ref = oracle.sgemm(A.numpy(), B.numpy())
        assert_close(run(tg, A, B, path=path), ref, K, f"{path} {M}x{N}x{K}")


@pytest.mark.parametrize("path", ["tf32x3", "ffma", "tiled", "tf32bf16"])
def test_integer_random_shapes_bitexact(tg, path):
    rng = np.random.default_rng(8)
    for i in range(6):
        M, N, K = (int(v) for v in rng.integers(1, 400, size=3))
        A, B = make_inputs(M, N, K, "int", 600 + i)
        ref = oracle.sgemm(A.numpy(), B.numpy())
        for split in (0, 1, 3):
            assert_bitexact(run(tg, A, B, path=path, split_k=split), ref, f"{path} {M}x{N}x{K} s{split}")


@pytest.mark.parametrize("path", ["tf32x3", "ffma", "tiled", "tf32bf16"])
@pytest.mark.parametrize("split", [0, 1, 2])
def test_strided_unaligned_views_and_canaries(tg, path, split):
    """Odd leading dimensions, unaligned base pointers (sub-views at odd
    offsets), and sentinel guard bands around C: nothing outside the M x N
    block of C may change."""
    M, N, K = 190, 263, 77
    lda, ldb, ldc = K + 3, N + 1, N + 5
    A, B = make_inputs(M, N, K, "uniform", 42)
    ref = oracle.sgemm(A.numpy(), B.numpy())
    dev = torch.device("cuda")
    Abuf = torch.zeros(1 + M * lda, device=dev)
    Bbuf = torch.zeros(3 + K * ldb, device=dev)
    Av = Abuf[1:].view(M, lda)[:, :K]
    Av.copy_(A.to(dev))
    Bv = Bbuf[3:].view(K, ldb)[:, :N]
    Bv.copy_(B.to(dev))
    guard = 1024
    Cbuf = torch.empty(2 * guard + 2 + M * ldc, device=dev)
    fill_sentinel(Cbuf)
    Cv = Cbuf[guard + 2: guard + 2 + M * ldc].view(M, ldc)[:, :N]
    tg.matmul(Av, Bv, out=Cv, path=path, split_k=split)
    torch.cuda.synchronize()
    assert tg.sync_status() == 0
    host = Cbuf.cpu().numpy()
    inside = np.zeros(host.shape, bool)
    idx = guard + 2 + (np.arange(M)[:, None] * ldc + np.arange(N)[None, :])
    inside[idx.ravel()] = True
    assert np.all(is_sentinel(host[~inside])), "write outside the M x N block of C"
    assert_close(host[idx], ref, K, f"strided {path}")


def test_k_zero_and_empty(tg):
    dev = torch.device("cuda")
    for path in ("tf32x3", "ffma", "tiled", "tf32bf16"):
        C = torch.empty(5, 7, device=dev)
        fill_sentinel(C)
        tg.matmul(torch.empty(5, 0, device=dev), torch.empty(0, 7, device=dev), out=C, path=path)
        torch.cuda.synchronize()
        assert np.all(C.cpu().numpy().view(np.uint32) == 0), "K = 0 must give +0.0"
        # M = 0 and N = 0 are no-ops
        tg.matmul(torch.empty(0, 4, device=dev), torch.empty(4, 3, device=dev), path=path)
        tg.matmul(torch.empty(4, 4, device=dev), torch.empty(4, 0, device=dev), path=path)
    assert tg.sync_status() == 0


def test_nan_row_propagates(tg):
    M, N, K = 40, 50, 60
    A, B = make_inputs(M, N, K, "uniform", 9)
    A[3, 17] = float("nan")
    ref = oracle.sgemm(A.numpy(), B.numpy())
    assert np.all(np.isnan(ref[3]))
    for path in ("tf32x3", "ffma", "tiled", "tf32bf16"):
        C = run(tg, A, B, path=path)
        assert np.all(np.isnan(C[3])), path
        keep = np.arange(M) != 3
        assert_close(C[keep], ref[keep], K, f"nan row {path}")


@pytest.mark.parametrize("path", ["tf32x3", "ffma", "tiled", "tf32bf16"])
def test_operands_near_float_max(tg, path):
    """Finite operands within 2^-11 of the largest float, times small ones:
    every product and sum is finite, so C must be too.  Rounding such a value
    to tf32 (or bf16) to nearest would carry it to infinity; the split
    truncates it instead."""
    M, N, K = 130, 260, 40
    rng = np.random.default_rng(77)
    fmax = np.finfo(np.float32).max
    A = (rng.uniform(0.9996, 1.0, (M, K)) * fmax * rng.choice([-1.0, 1.0], (M, K))).astype(np.float32)
    A[:, ::3] = rng.uniform(-1, 1, (M, (K + 2) // 3)).astype(np.float32)  # mixed with ordinary values
    B = (rng.uniform(-1, 1, (K, N)) * 2.0 ** -100).astype(np.float32)
    # large values in A (split row by row) and, transposed, in B (split by the
    # transposing pass)
    for X, Y in [(A, B), (np.ascontiguousarray(B.T), np.ascontiguousarray(A.T))]:
        X, Y = torch.from_numpy(X), torch.from_numpy(Y)
        ref = oracle.sgemm(X.numpy(), Y.numpy())
        assert np.all(np.isfinite(ref))
        C = run(tg, X, Y, path=path)
        assert np.all(np.isfinite(C)), path
        assert_close(C, ref, K, f"near FLT_MAX {path} {tuple(X.shape)}")


def test_deterministic(tg):
    A, B, _, _ = workload_case("ragged_777x1029x513")
    for path in ("tf32x3", "ffma", "tiled", "tf32bf16"):
        c1 = run(tg, A, B, path=path)
        c2 = run(tg, A, B, path=path)
        assert np.array_equal(c1.view(np.uint32), c2.view(np.uint32)), path


def test_caller_workspace(tg):
    A, B, _, ref = workload_case("ragged_777x1029x513")
    Ad, Bd = A.cuda(), B.cuda()
    C = torch.empty(A.shape[0], B.shape[1], device="cuda")
    need = tg.plan(A.shape[0], B.shape[1], A.shape[1], A=Ad.data_ptr(), B=Bd.data_ptr(),
                   C=C.data_ptr(), path="tf32x3")["workspace_bytes"]
    ws = torch.empty(need // 4 + 64, device="cuda")
    tg.matmul(Ad, Bd, out=C, path="tf32x3", workspace=ws)
    torch.cuda.synchronize()
    assert_close(C.cpu().numpy(), ref, A.shape[1], "caller workspace")
    small = torch.empty(16, device="cuda")
    with pytest.raises(tg.TgError) as e:
        tg.matmul(Ad, Bd, out=C, path="tf32x3", workspace=small)
    assert e.value.status == 6


def test_host_buffer_entry(tg):
    """A small product is one block: bit-identical to tg_sgemm on the same
    device layout (the host entry copies A into rows padded to 16 bytes, which
    the GEMM kernel splits itself; lda = 513 would take the pre-pass)."""
    A, B, _, ref = workload_case("ragged_777x1029x513")
    Ap, Bp = A.pin_memory(), B.pin_memory()
    C = torch.empty(A.shape[0], B.shape[1]).pin_memory()
    tg.sgemm_host(Ap, Bp, C)
    assert_close(C.numpy(), ref, A.shape[1], "host entry")
    M, K = A.shape
    Apad = torch.zeros(M, -(-K // 4) * 4, device="cuda")
    Apad[:, :K] = A.cuda()
    dev = tg.matmul(Apad[:, :K], B.cuda())
    torch.cuda.synchronize()
    assert np.array_equal(C.numpy().view(np.uint32), dev.cpu().numpy().view(np.uint32))


@pytest.mark.parametrize("path", ["tf32x3", "ffma", "tf32bf16"])
def test_host_buffer_entry_row_blocks(tg, path):
    """A product large enough for the host entry point to pipeline row blocks
    (copies of one block overlapping the product of another), with a ragged
    last block and padded host rows; checked on sampled rows."""
    M, N, K = 4100, 1030, 2050
    A, B = make_inputs(M, N, K, "uniform", 321)
    Abig = torch.zeros(M, K + 3)
    Abig[:, :K] = A
    Ap = Abig.pin_memory()[:, :K]
    Bp = B.pin_memory()
    Cbig = torch.full((M, N + 5), float("nan")).pin_memory()
    C = Cbig[:, :N]
    tg.sgemm_host(Ap, Bp, C, path=path)
    rows = np.sort(np.random.default_rng(3).choice(M, 200, replace=False))
    rows = np.unique(np.concatenate([rows, [0, 1151, 1152, 2303, 2304, M - 1]]))
    ref = oracle.sgemm_rows(A.numpy(), B.numpy(), rows)
    assert_close(C.numpy()[rows], ref, K, f"host row blocks {path}")
    assert np.all(np.isnan(Cbig.numpy()[:, N:])), "host entry wrote past column N"


@pytest.mark.parametrize("layout", [None, "1024,1024,1536,4", "512,1536,1024,2,1"])
@pytest.mark.parametrize("path", ["tf32x3", "ffma", "tf32bf16"])
def test_host_buffer_entry_2d_blocks(tg, path, layout, monkeypatch):
    """The host entry point with C cut into row blocks, the first ones also
    into column blocks (ragged last ones), the later ones full width: every
    product waits for its own A row block and B column block (all of B when
    full width), A and B are split once and reused, C blocks are copied out
    as they finish (or after the last copy in).  The model's layout, every
    row block cut, and two of four cut with the copies out held back.
    Sampled rows at and around every row-block edge, all columns."""
    if layout is not None:
        monkeypatch.setenv("TG_HOST_BLOCKS", layout)
    M, N, K = 4100, 3000, 1500
    hb = tg.host_blocks(M, N, K, path=path)
    assert hb["row_blocks"] > 1
    if layout is not None:
        assert hb["col_blocks"] > 1
        fields = ("first_block_rows", "block_rows", "block_cols", "split_row_blocks", "defer_copies_out")
        want = [int(x) for x in layout.split(",")]
        assert [hb[k] for k in fields[:len(want)]] == want
    A, B = make_inputs(M, N, K, "uniform", 322)
    Ap, Bp = A.pin_memory(), B.pin_memory()
    Cbig = torch.full((M, N + 3), float("nan")).pin_memory()
    C = Cbig[:, :N]
    tg.sgemm_host(Ap, Bp, C, path=path)
    f, mb = hb["first_block_rows"], hb["block_rows"]
    edges = [r for i in range(1, hb["row_blocks"]) for r in (f + (i - 1) * mb - 1, f + (i - 1) * mb)]
    rows = np.sort(np.random.default_rng(4).choice(M, 120, replace=False))
    rows = np.unique(np.concatenate([rows, [0, M - 1], edges]))
    ref = oracle.sgemm_rows(A.numpy(), B.numpy(), rows)
    assert_close(C.numpy()[rows], ref, K, f"host 2-D blocks {path}")
    assert np.all(np.isnan(Cbig.numpy()[:, N:])), "host entry wrote past column N"
    dev = run(tg, A, B, path=path)  # same products as the device entry, block by block
    assert_close(C.numpy(), dev, K, f"host vs device {path}")


def test_host_trace_timeline(tg):
    """TG_HOST_TRACE=1 prints the host call's timeline: every copy in, every
    product's begin and end and every copy out, with times that start at 0
    and products that end after they begin."""
    import re
    import subprocess
    import sys

    code = ("import numpy as np, torch, shared_memory_tiled_fp32_gb300 as tg;"
            "A = torch.ones(4100, 1500).pin_memory(); B = torch.ones(1500, 3000).pin_memory();"
            "C = torch.empty(4100, 3000).pin_memory(); tg.sgemm_host(A, B, C);"
            "assert float(C[0, 0]) == 1500.0 and float(C[-1, -1]) == 1500.0")
    env = dict(os.environ, TG_HOST_TRACE="1", TG_HOST_BLOCKS="1024,1024,1536,2,1")
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=300,
                       cwd=os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stderr.splitlines() if ln.startswith("tg_host_trace")]
    times = {m.group(2): float(m.group(1)) for m in
             (re.match(r"tg_host_trace\s+([0-9.]+) ms (.*)$", ln) for ln in lines) if m}
    # 5 row blocks: the first two cut into 2 column blocks, the other three full width
    assert sum(k.startswith("in A") for k in times) == 5 and sum(k.startswith("in B") for k in times) == 2
    products = [k[len("product "):-len(" begins")] for k in times if k.endswith(" begins")]
    assert len(products) == 2 * 2 + 3
    for p in products:
        assert times[f"product {p} ends"] >= times[f"product {p} begins"] >= 0.0
        assert times[f"out {p}"] >= times[f"product {p} ends"]
    # copies out held back until the last copy in
    assert min(times[f"out {p}"] for p in products) >= max(v for k, v in times.items() if k.startswith("in "))


def test_side_stream(tg):
    A, B, _, ref = workload_case("sq256_uniform")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        Ad, Bd = A.cuda(), B.cuda()
        C = tg.matmul(Ad, Bd, stream=s)
    s.synchronize()
    assert_close(C.cpu().numpy(), ref, A.shape[1], "side stream")


def test_plan_on_device(tg):
    p = tg.plan(8192, 8192, 8192)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert p["grid"] == min(p["units"], sms)
    assert p["path"] == "tf32x3"


@pytest.mark.parametrize("path", ["tf32x3", "tf32bf16"])
@pytest.mark.parametrize("pair,pair_mma", [("0", "1"), ("1", "0"), ("1", "1")])
def test_tf32x3_cluster_pairs_on_and_off(tg, pair, pair_mma, path, monkeypatch):
    """The three forms of the 3xTF32 kernel: one CTA per tile; CTA pairs with
    one M = 128 product per CTA, each CTA loading the whole B tile; CTA pairs with one
    M = 256 product over both (cta_group::2, each CTA holding its half of B)
    -- including odd tile-row counts (the last pair's second CTA is all
    ghost), split K and a stream-K tail."""
    monkeypatch.setenv("TG_TF32X3_PAIR", pair)
    monkeypatch.setenv("TG_TF32X3_PAIRMMA", pair_mma)
    for i, (M, N, K) in enumerate([(129, 300, 700), (383, 513, 300), (640, 256, 2048), (1, 7, 9),
                                   (1000, 3000, 1100)]):
        A, B = make_inputs(M, N, K, "uniform", 900 + i)
        ref = oracle.sgemm(A.numpy(), B.numpy())
        p = tg.plan(M, N, K, path=path)
        assert p["tiles_m"] == -(-M // 128) and p["path"] == path
        for split in (0, 1, 2):
            assert_close(run(tg, A, B, path=path, split_k=split), ref, K,
                         f"{path} pair={pair} mma={pair_mma} {M}x{N}x{K} s{split}")
    A, B = make_inputs(1000, 3000, 1100, "int", 911)
    assert_bitexact(run(tg, A, B, path=path), oracle.sgemm(A.numpy(), B.numpy()), f"{path} pair forms, integers")


TAIL_CASES = [(1000, 3000, 1100, "uniform", "tf32x3"), (1000, 3000, 1100, "int", "tf32x3"),
              (4000, 3900, 8000, "uniform", "tf32x3"), (400, 8000, 20000, "normal", "tf32x3"),
              (400, 8000, 20000, "int", "tf32x3"), (1000, 3000, 1100, "uniform", "tf32bf16"),
              (400, 8000, 20000, "int", "tf32bf16"), (1000, 3000, 1100, "uniform", "ffma"),
              (1000, 3000, 1100, "int", "ffma"), (400, 8000, 20000, "normal", "ffma")]


@pytest.mark.parametrize("M,N,K,dist,path", TAIL_CASES)
def test_balanced_tail(tg, M, N, K, dist, path):
    """Shapes whose last round is shared out over more lanes than it has units
    (pieces of a unit added by the tail reduce in lane order), with ragged
    edges: stream-K runs on both paths, with fewer units than lanes and runs
    shorter than a unit (some units spread over three lanes); equal K slices
    on the 3xTF32 path when the tail's rows exceed L2 (4000 x 3900 x 8000),
    or a split point when such a tail fills more than half the lanes
    (400 x 8000 x 20000: every unit's first K blocks on its own lane, the
    rest spread over the others).  Every output is checked; integer inputs
    bit-exactly."""
    A, B = make_inputs(M, N, K, dist, 700 + K % 97)
    p = tg.plan(M, N, K, path=path)
    assert p["tail_units"] > 0 and p["tail_lanes"] > p["tail_units"]
    ref = oracle.sgemm(A.numpy(), B.numpy())
    got = run(tg, A, B, path=path)
    if dist == "int":
        assert_bitexact(got, ref, f"stream-K {path} {M}x{N}x{K}")
    else:
        assert_close(got, ref, K, f"stream-K {path} {M}x{N}x{K}")
    again = run(tg, A, B, path=path)  # the fixed-order reduce gives the same bits
    assert np.array_equal(got.view(np.uint32), again.view(np.uint32))


@pytest.mark.parametrize("path,M,N,K", [("tf32x3", 1000, 3000, 1100), ("ffma", 1000, 3000, 1100),
                                        ("tf32x3", 400, 8000, 20000), ("tf32x3", 4000, 3900, 8000)])
def test_balanced_tail_scaled(tg, path, M, N, K):
    """alpha and beta on balanced last rounds (stream-K, split point, equal K
    slices): applied by the GEMM epilogue for units one lane ran whole and by
    the tail reduce for the others."""
    A, B = make_inputs(M, N, K, "uniform", 731)
    C0 = np.random.default_rng(732).uniform(-1, 1, (M, N)).astype(np.float32)
    Cd = torch.from_numpy(C0.copy()).cuda()
    tg.matmul_general(A.cuda(), B.cuda(), Cd, alpha=0.5, beta=-1.5, path=path)
    torch.cuda.synchronize()
    assert tg.sync_status() == 0
    ref = oracle.sgemm_general(0, 0, 0.5, A.numpy(), B.numpy(), -1.5, C0.copy())
    assert_close(Cd.cpu().numpy(), ref, K, f"balanced tail scaled {path} {M}x{N}x{K}")


@pytest.mark.parametrize("path", ["tf32x3", "ffma", "tf32bf16"])
@pytest.mark.parametrize("M,N,K", [(3, 5, 1 << 22), (2, 1 << 24, 3), (1 << 22, 7, 9)])
def test_extreme_aspect_ratios(tg, path, M, N, K):
    """Products of hundreds of MB with one dimension in the millions and the
    others tiny: a K split over 2^18 K blocks, 65,536 tile columns, 32,768
    tile rows (64-bit tile and row offsets, ghost-heavy edge tiles), every
    output checked against the oracle."""
    A, B = make_inputs(M, N, K, "uniform", 40 + (M % 7))
    C = run(tg, A, B, path=path)
    ref = oracle.sgemm(A.numpy(), B.numpy())  # at most 2^25 outputs, 2^28 multiply-adds
    assert_close(C, ref, K, f"{M}x{N}x{K} {path}")


@pytest.mark.parametrize("M,N,K", [(777, 1029, 513), (2048, 2048, 4096), (256, 256, 256)])
def test_cuda_graph_capture_and_replay(tg, M, N, K):
    """A call captured into a CUDA graph (workspace from the stream-ordered
    pool becomes graph memory, the launches keep their programmatic
    dependencies) and replayed on new inputs gives the same bits as the
    eager call on those inputs."""
    A0, B0 = make_inputs(M, N, K, "uniform", 61)
    A1, B1 = make_inputs(M, N, K, "normal", 62)
    Ad, Bd = A0.cuda(), B0.cuda()
    C = torch.empty(M, N, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        tg.matmul(Ad, Bd, out=C, stream=s)  # first use of the device state outside the capture
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        tg.matmul(Ad, Bd, out=C, stream=s)
    for A, B in ((A1, B1), (A0, B0)):
        Ad.copy_(A)
        Bd.copy_(B)
        C.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert tg.sync_status() == 0
        eager = run(tg, A, B)
        assert np.array_equal(C.cpu().numpy().view(np.uint32), eager.view(np.uint32))
