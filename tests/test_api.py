"""Host-side checks of the C ABI that need no GPU: the library loads, exports
every symbol the header declares, rejects bad arguments before touching CUDA,
and plans tiles, K splits and workspace as documented."""
import ctypes
import os
import re

import pytest

import shared_memory_tiled_fp32_gb300 as tg
from shared_memory_tiled_fp32_gb300 import binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", h) for h in sorted(os.listdir(os.path.join(ROOT, "include")))
           if h.endswith(".h")]


def header_functions():
    src = "".join(open(h).read() for h in HEADERS)
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?(?:unsigned\s+)?[a-z_]+\s*\**\s*(tg_\w+)\s*\(", src, flags=re.M)))


def test_library_exports_header_symbols():
    L = tg.lib()
    funcs = header_functions()
    assert funcs, "no declarations parsed"
    assert sorted(binding.EXPORTS) == funcs
    for name in funcs:
        assert hasattr(L, name), name


def test_version_and_status_strings():
    assert tg.lib().tg_sgemm_version() == 100
    for code, name in tg.STATUS.items():
        assert tg.status_string(code).startswith(name)


def _call(M, N, K, A, lda, B, ldb, C, ldc, path=0, split=0):
    o = binding.Opts()
    o.path, o.split_k = path, split
    return tg.lib().tg_sgemm_ex(M, N, K, A, lda, B, ldb, C, ldc, None, ctypes.byref(o))


def test_argument_errors_need_no_gpu():
    p = 1 << 20  # never dereferenced: every case below fails validation first
    bad = [
        (-1, 4, 4, p, 4, p + 10**6, 4, p + 2 * 10**6, 4),
        (4, -1, 4, p, 4, p + 10**6, 4, p + 2 * 10**6, 4),
        (4, 4, -1, p, 4, p + 10**6, 4, p + 2 * 10**6, 4),
        (4, 4, 8, p, 7, p + 10**6, 4, p + 2 * 10**6, 4),     # lda < K
        (4, 8, 4, p, 4, p + 10**6, 7, p + 2 * 10**6, 8),     # ldb < N
        (4, 8, 4, p, 4, p + 10**6, 8, p + 2 * 10**6, 7),     # ldc < N
        (4, 4, 4, None, 4, p + 10**6, 4, p + 2 * 10**6, 4),  # null A
        (4, 4, 4, p, 4, None, 4, p + 2 * 10**6, 4),          # null B
        (4, 4, 4, p, 4, p + 10**6, 4, None, 4),              # null C
        (4, 4, 4, p, 4, p + 10**6, 4, p + 8, 4),             # C overlaps A
        (4, 4, 4, p, 4, p + 10**6, 4, p + 10**6 + 60, 4),    # C overlaps B
    ]
    for args in bad:
        assert _call(*args) == 1, args
    assert _call(4, 4, 4, p, 4, p + 10**6, 4, p + 2 * 10**6, 4, path=7) == 1
    assert _call(4, 4, 4, p, 4, p + 10**6, 4, p + 2 * 10**6, 4, split=-2) == 1
    # empty outputs are a valid no-op that never reaches the device
    assert _call(0, 4, 4, None, 4, None, 4, None, 4) == 0
    assert _call(4, 0, 4, None, 4, None, 1, None, 1) == 0


def test_plan_tiles_split_and_workspace():
    sms = 152
    p = tg.plan(8192, 8192, 8192, num_sms=sms)
    assert (p["path"], p["tiles_m"], p["tiles_n"], p["split_k"]) == ("tf32x3", 64, 32, 1)
    # pairs of vertically adjacent tiles share B (cluster of 2 CTAs); 1024 pair
    # units on 76 pairs leave 36 for a last round, which is cut into 2 K slices
    assert p["pair"] == 2 and p["grid"] == sms and p["launches"] == 3
    assert (p["tail_units"], p["tail_split"]) == (36, 2)
    assert p["units"] == (32 * 32 - 36) + 36 * 2
    # A_hi, A_lo, B_hi^T, B_lo^T, plus the tail partials: 36 units x 2 slices x 256 x 256
    assert p["workspace_bytes"] == 4 * 8192 * 8192 * 4 + 36 * 2 * 256 * 256 * 4
    # an explicit split turns the last-round balancing off
    q = tg.plan(8192, 8192, 8192, num_sms=sms, split_k=1)
    assert q["tail_units"] == 0 and q["units"] == 1024 and q["launches"] == 2
    # ragged: ceil(777/128) x ceil(1029/256) tiles, split to fill the SMs
    p = tg.plan(777, 1029, 513, num_sms=sms)
    assert (p["tiles_m"], p["tiles_n"]) == (7, 5)
    assert p["split_k"] == 4 and p["pair"] == 2 and p["units"] == 4 * 5 * 4 and p["launches"] == 3
    assert p["grid"] == 2 * min(p["units"], sms // 2)
    # one tile row cannot be paired; FFMA never pairs
    assert tg.plan(100, 4096, 4096, num_sms=sms)["pair"] == 1
    assert tg.plan(4096, 4096, 4096, num_sms=sms, path="ffma")["pair"] == 1
    # an explicit split is capped by the K blocks
    p = tg.plan(64, 64, 32, num_sms=sms, split_k=9)
    assert p["split_k"] == 2  # ceil(32/16) K blocks
    # FFMA reads aligned operands in place and packs misaligned ones
    one = dict(num_sms=sms, path="ffma", split_k=1)
    a = tg.plan(512, 512, 512, A=4096, B=1 << 20, C=1 << 24, **one)
    assert a["prepass"] == 0 and a["workspace_bytes"] == 0 and a["launches"] == 1
    b = tg.plan(512, 512, 512, A=4100, B=1 << 20, C=1 << 24, **one)
    assert b["prepass"] == 1 and b["workspace_bytes"] == 512 * 512 * 4 and b["launches"] == 2
    c = tg.plan(512, 513, 512, 512, 513, 513, A=4096, B=1 << 20, C=1 << 24, **one)
    assert c["prepass"] == 1 and c["workspace_bytes"] == 512 * 516 * 4
    # few tiles: K is split so the SMs fill, partials add 4 * S * M * roundup(N, 4) bytes
    d = tg.plan(512, 512, 512, A=4096, B=1 << 20, C=1 << 24, num_sms=sms, path="ffma")
    assert d["split_k"] == 4 and d["workspace_bytes"] == 4 * 4 * 512 * 512 and d["launches"] == 2
    # K = 0 is one fill kernel
    z = tg.plan(10, 10, 0, num_sms=sms)
    assert z["launches"] == 1 and z["workspace_bytes"] == 0


@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (300, 7, 5000), (2048, 2048, 16384), (129, 257, 17)])
def test_plan_split_ranges_cover_k(M, N, K):
    """Each K slice gets a non-empty, contiguous run of K blocks."""
    for path in ("tf32x3", "ffma"):
        p = tg.plan(M, N, K, num_sms=152, path=path)
        nkb = -(-K // p["block_k"])
        S = p["split_k"]
        bounds = [s * nkb // S for s in range(S + 1)]
        assert bounds[0] == 0 and bounds[-1] == nkb
        assert all(b1 > b0 for b0, b1 in zip(bounds, bounds[1:]))


def _general(opa, opb, M, N, K, lda, ldb, ldc, A=1 << 20, B=1 << 32, C=1 << 36):
    o = binding.Opts()
    return tg.lib().tg_sgemm_general(opa, opb, M, N, K, 1.0, A, lda, B, ldb, 0.0, C, ldc, None, ctypes.byref(o))


def test_general_argument_errors_need_no_gpu():
    # stored shapes: A is K x M for op T (lda >= M); B is N x K for op T (ldb >= K)
    assert _general(1, 0, 8, 4, 6, 7, 4, 4) == 1   # op T: lda < M
    assert _general(0, 1, 8, 4, 6, 6, 5, 4) == 1   # op T: ldb < K
    assert _general(2, 0, 8, 4, 6, 8, 4, 4) == 1   # bad op
    assert _general(0, -1, 8, 4, 6, 8, 4, 4) == 1
    # C overlapping a transposed A: A spans K rows of lda
    assert _general(1, 0, 8, 4, 6, 8, 4, 4, A=1 << 20, C=(1 << 20) + 4 * 8 * 5) == 1
    assert _general(1, 0, 0, 4, 6, 8, 4, 4) == 0   # empty output: no-op, no device touched


def test_general_plan_packs_transposed_operands():
    sms = 152
    one = dict(num_sms=sms, path="ffma", split_k=1, A=4096, B=1 << 20, C=1 << 24)
    # FFMA reads untransposed, aligned operands in place; a transposed one is packed
    assert tg.plan_general(0, 0, 512, 512, 512, 512, 512, 512, **one)["prepass"] == 0
    pa = tg.plan_general(1, 0, 512, 512, 256, 512, 512, 512, **one)
    assert pa["prepass"] == 1 and pa["workspace_bytes"] == 512 * 256 * 4
    pb = tg.plan_general(0, 1, 512, 768, 256, 256, 256, 768, **one)
    assert pb["prepass"] == 1 and pb["workspace_bytes"] == 256 * 768 * 4
    # 3xTF32 always re-lays both operands; the workspace does not depend on ops
    t = [tg.plan_general(a, b, 777, 1029, 513, 777 if a else 513, 513 if b else 1029, 1029, num_sms=sms)
         for a in (0, 1) for b in (0, 1)]
    assert len({x["workspace_bytes"] for x in t}) == 1

