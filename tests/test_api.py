"""Host-side checks of the C ABI that need no GPU: the library loads, exports
every symbol the header declares, rejects bad arguments before touching CUDA,
and plans tiles, K splits and workspace as documented."""
import ctypes
import os
import re

import numpy as np
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
    assert tg.lib().tg_sgemm_version() == 103
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
    # units on 76 pairs leave 36 after 13 whole rounds.  Their A and B rows
    # (groups of 19 pair rows: the last 36 units are 3 columns of the second
    # group's 13 pair rows, 3328 rows + 768 columns of K = 8192, hi and lo)
    # exceed L2, so each is cut into 2 equal K slices: 72 lanes, half a round
    assert p["pair"] == 2 and p["grid"] == sms and p["launches"] == 3
    assert (p["tail_units"], p["tail_lanes"]) == (36, 72)
    assert p["units"] == 32 * 32
    # A_hi, A_lo, B_hi^T, B_lo^T, plus two partial slots of 256 x 256 per lane
    assert p["workspace_bytes"] == 4 * 8192 * 8192 * 4 + 2 * 72 * 256 * 256 * 4
    # 4096^3: the 28-unit tail (the last two columns of one group of all 16
    # pair rows) reads all 4096 rows of A and 512 columns of B.  Split by the
    # pre-pass (no A given: 8 bytes per element) that is 150 MB, past L2 ->
    # 2 equal K slices, 56 lanes; A split in the kernel (4 bytes) 84 MB ->
    # stream-K over all 76 pairs
    m = tg.plan(4096, 4096, 4096, num_sms=sms)
    assert (m["units"], m["tail_units"], m["tail_lanes"]) == (256, 28, 56)
    m = tg.plan(4096, 4096, 4096, A=1 << 40, B=2 << 40, C=3 << 40, num_sms=sms)
    assert m["fused_split"] == 1
    assert (m["units"], m["tail_units"], m["tail_lanes"]) == (256, 28, 76)
    # an explicit split turns the tail balancing off
    q = tg.plan(8192, 8192, 8192, num_sms=sms, split_k=1)
    assert q["tail_units"] == 0 and q["units"] == 1024 and q["launches"] == 2
    # long K, fewer units than lanes: FFMA (128 units, 152 CTAs) runs all of it
    # stream-K on every CTA
    lk = tg.plan(2048, 2048, 16384, num_sms=sms, path="ffma")
    assert (lk["units"], lk["tail_units"], lk["tail_lanes"], lk["grid"]) == (128, 128, 152, sms)
    lt = tg.plan(2048, 2048, 16384, num_sms=sms)
    # 3xTF32 (64 pair units, rows far past L2, more than half the lanes):
    # split point, lane q runs the first 862 of unit q's 1024 K blocks in step
    # with the others, the 12 remaining pairs share the rest
    assert (lt["units"], lt["tail_units"], lt["tail_lanes"], lt["tail_kx"], lt["grid"]) == (64, 64, 76, 862, sms)
    # a tail that fills 90 % of a round or more is left alone
    assert tg.plan(128 * 2 * 70, 256, 4096, num_sms=sms)["tail_units"] == 0
    # a short K gives too little work per lane to share out
    assert tg.plan(4096, 4096, 128, num_sms=sms)["tail_units"] == 0
    # ragged: ceil(777/128) x ceil(1029/256) tiles = 4 pair rows x 5 columns,
    # K split to fill one round of the 76 pairs without a second: 3 slices
    p = tg.plan(777, 1029, 513, num_sms=sms)
    assert (p["tiles_m"], p["tiles_n"]) == (7, 5)
    assert p["split_k"] == 3 and p["pair"] == 2 and p["units"] == 4 * 5 * 3 and p["launches"] == 3
    assert p["units"] <= sms // 2 and p["grid"] == 2 * p["units"]
    # every automatic K split keeps its units within one round of the lanes
    for (M, N, K) in [(777, 1029, 513), (300, 300, 3000), (1024, 1024, 8192), (1500, 600, 2000), (129, 4000, 900)]:
        for path in ("tf32x3", "ffma"):
            q = tg.plan(M, N, K, num_sms=sms, path=path)
            if q["split_k"] > 1:
                assert q["units"] <= sms // q["pair"], (M, N, K, path, q)
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
    # small products: the tiled path (64 x 64 tiles, operands in place, no
    # pre-pass, one launch, no workspace).  16 tiles would leave most SMs
    # idle, so K is split into 8 slices of two 16-wide stages: a cluster of 8
    # blocks per tile adds the slices in shared memory (128 blocks)
    t = tg.plan(256, 256, 256, num_sms=sms)
    assert (t["path"], t["tiles_m"], t["tiles_n"], t["split_k"], t["grid"], t["launches"], t["prepass"],
            t["workspace_bytes"]) == ("tiled", 4, 4, 8, 128, 1, 0, 0)
    # a short K (fewer than 8 blocks of 16) is not split
    assert tg.plan(100, 100, 100, num_sms=sms)["split_k"] == 1
    # an explicit split on the tiled path is honoured, at most 8 (one cluster)
    v = tg.plan(200, 300, 100, num_sms=sms, path="tiled", split_k=3)
    assert (v["split_k"], v["grid"], v["launches"]) == (3, 4 * 5 * 3, 1)
    assert tg.plan(200, 300, 1000, num_sms=sms, path="tiled", split_k=12)["split_k"] == 8
    assert tg.plan(256, 256, 256, num_sms=sms, split_k=2)["path"] == "tf32x3"
    assert tg.plan(512, 512, 512, num_sms=sms)["path"] == "tf32x3"    # 2^27 multiply-adds
    assert tg.plan(64, 64, 8192, num_sms=sms)["path"] == "tf32x3"     # long K: split instead
    assert tg.plan(777, 1029, 513, num_sms=sms, path="tiled")["tiles_m"] == 13
    # the tf32 + bf16 cross-product path only on request, with the 3xTF32
    # tiles, workspace and launches (its split tiles have the same size)
    for shape in [(8192, 8192, 8192), (777, 1029, 513), (4000, 3900, 8000), (64, 64, 8192)]:
        x, m = tg.plan(*shape, num_sms=sms, path="tf32x3"), tg.plan(*shape, num_sms=sms, path="tf32bf16")
        assert m["path"] == "tf32bf16" and tg.plan(*shape, num_sms=sms)["path"] != "tf32bf16"
        assert {k: v for k, v in m.items() if k != "path"} == {k: v for k, v in x.items() if k != "path"}


def _split_point_pieces(U, nkb, L, kx, slots):
    """The split-point tail as the 3xTF32 kernel walks it: lane q < U runs the
    first kx K blocks of unit q (slot q*slots); the other E = L - U lanes run
    the remaining blocks of all units laid end to end, one piece per unit
    they meet (slot q*slots + 1 + i, i counted from the first lane meeting
    unit q's remainder)."""
    E, rl = L - U, nkb - kx
    R = U * rl
    lane_of = lambda x: ((x + 1) * E + R - 1) // R - 1
    for q in range(U):
        yield q, q, 0, kx, q * slots
    for e in range(E):
        s, t = e * R // E, (e + 1) * R // E
        q = s // rl
        while s < t and q * rl < t:
            b0 = q * rl
            lo, hi = max(s, b0) - b0, min(t, b0 + rl) - b0
            yield U + e, q, kx + lo, kx + hi, q * slots + 1 + (e - lane_of(b0))
            q += 1


@pytest.mark.parametrize("M,N,K", [(2048, 2048, 16384), (400, 8000, 20000)])
def test_split_point_tail_covers_every_unit_once(M, N, K):
    """Host model of the split-point tail (3xTF32 tails larger than L2 that
    fill more than half the lanes): every K block of every tail unit runs
    exactly once, the lockstep first parts and the remainder pieces give every
    lane a similar share, and no two pieces share a partial slot."""
    p = tg.plan(M, N, K, num_sms=152)
    U, L, kx, nkb = p["tail_units"], p["tail_lanes"], p["tail_kx"], -(-K // p["block_k"])
    assert kx > 0 and U < L and 10 * kx <= 9 * nkb
    E = L - U
    rl = nkb - kx
    share = U * rl // E
    slots = 1 + -(-rl // share) + 1
    pieces = list(_split_point_pieces(U, nkb, L, kx, slots))
    covered = np.zeros((U, nkb), np.int32)
    used = set()
    work = np.zeros(L, np.int64)
    for lane, q, lo, hi, slot in pieces:
        assert 0 <= lo < hi <= nkb and slot not in used and q * slots <= slot < (q + 1) * slots
        used.add(slot)
        covered[q, lo:hi] += 1
        work[lane] += hi - lo
    assert np.all(covered == 1)
    assert work.max() - work.min() <= max(2, nkb // 50)  # balanced lanes
    assert U * slots * p["pair"] * p["block_m"] * p["block_n"] * 4 <= p["workspace_bytes"]


def _tail_pieces(tail_units, nkb, lanes):
    """The stream-K tail as the GEMM kernels walk it: lane v runs K blocks
    [v*T/lanes, (v+1)*T/lanes) of the T = tail_units * nkb blocks laid end to
    end, one piece per tail unit it meets; a piece short of its whole unit
    writes partial slot 2v (the lane's first piece) or 2v + 1 (its last)."""
    T = tail_units * nkb
    for v in range(lanes):
        s, e = v * T // lanes, (v + 1) * T // lanes
        q = q0 = s // nkb
        while q * nkb < e and s < e:
            lo, hi = max(s, q * nkb) - q * nkb, min(e, (q + 1) * nkb) - q * nkb
            direct = lo == 0 and hi == nkb
            yield v, q, lo, hi, None if direct else 2 * v + (0 if q == q0 else 1)
            q += 1


@pytest.mark.parametrize("M,N,K,path,sliced", [
    (8192, 8192, 8192, "tf32x3", True), (4000, 3900, 8000, "tf32x3", True), (4096, 4096, 4096, "tf32x3", False),
    (1000, 3000, 1100, "tf32x3", False), (8192, 8192, 8192, "ffma", False), (2048, 2048, 16384, "ffma", False),
    (400, 8000, 20000, "ffma", False)])
def test_tail_runs_cover_every_unit_once(M, N, K, path, sliced):
    """Host model of the balanced last round of a plan: every K block of
    every tail unit is run exactly once, a lane writes at most its two slots,
    and the reduce's lookup (lanes holding the unit's first to last K block,
    slot 2v when the unit is the lane's first) finds exactly the pieces
    written.  With equal K slices every run lies inside one unit."""
    p = tg.plan(M, N, K, num_sms=152, path=path)
    tu, L, nkb = p["tail_units"], p["tail_lanes"], -(-K // p["block_k"])
    assert tu > 0 and L > tu and 10 * tu <= 9 * L
    assert (p["units"] - tu) % (p["grid"] // p["pair"]) == 0 or p["units"] < L
    T = tu * nkb
    if sliced:
        assert L % tu == 0 and 2 <= L // tu <= 4 and nkb >= 8 * (L // tu)
    else:
        assert T // L >= 512 // p["block_k"]  # every lane's share is at least 512 of K
    pieces = list(_tail_pieces(tu, nkb, L))
    covered = np.zeros((tu, nkb), np.int32)
    slots = {}
    for v, q, lo, hi, slot in pieces:
        assert 0 <= lo < hi <= nkb
        covered[q, lo:hi] += 1
        if slot is not None:
            assert slot // 2 == v and slot not in slots
            slots[slot] = q
    assert np.all(covered == 1)
    lane_of = lambda x: ((x + 1) * L + T - 1) // T - 1
    for q in range(tu):
        v0, v1 = lane_of(q * nkb), lane_of((q + 1) * nkb - 1)
        mine = [pc for pc in pieces if pc[1] == q]
        assert [pc[0] for pc in mine] == list(range(v0, v1 + 1))
        if v0 == v1:
            assert mine[0][4] is None
        else:
            want = sorted(2 * v + (0 if (v * T // L) // nkb == q else 1) for v in range(v0, v1 + 1))
            assert sorted(pc[4] for pc in mine) == want and all(slots[w] == q for w in want)
    assert 2 * L * p["pair"] * p["block_m"] * p["block_n"] * 4 <= p["workspace_bytes"]
    if sliced:
        assert len(pieces) == L and all(slot in (None, 2 * v) for v, _, _, _, slot in pieces)


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



@pytest.mark.parametrize("M,N,K,path", [(8192, 8192, 8192, "tf32x3"), (8192, 8192, 8192, "ffma"),
                                        (4096, 4096, 4096, "tf32x3"), (2048, 2048, 16384, "tf32x3"),
                                        (4100, 1030, 2050, "tf32x3"), (777, 1029, 513, "ffma"), (1, 1, 1, "tf32x3"),
                                        (5000, 300, 0, "tf32x3")])
def test_host_blocks_cover_c(M, N, K, path):
    """The host entry's output blocks: rows in multiples of 128, columns in
    multiples of 256, exactly covering C (the last ones ragged), at most 8 row
    blocks, the first split_row_blocks of them cut into at most 8 column
    blocks."""
    h = tg.host_blocks(M, N, K, path=path, num_sms=152)
    pm, pn, f, mb, nb = h["row_blocks"], h["col_blocks"], h["first_block_rows"], h["block_rows"], h["block_cols"]
    split = h["split_row_blocks"]
    assert 1 <= pm <= 8 and 1 <= pn <= 8 and 1 <= split <= pm
    assert f % 128 == 0 and mb % 128 == 0 and nb % 256 == 0
    # row blocks: [0, f), then blocks of mb rows, the last one the remainder
    assert (pm == 1 and f >= M) or (pm > 1 and f < M and -(-(M - f) // mb) == pm - 1)
    assert -(-N // nb) == pn
    assert h["model_ms"] >= 0
    if pm > 1:
        assert mb >= 512
    if pn > 1:
        assert nb >= 512


def test_host_blocks_override(monkeypatch):
    """TG_HOST_BLOCKS fixes the layout when it describes valid blocks of C and
    is ignored otherwise."""
    model = tg.host_blocks(4100, 3000, 1500, path="tf32x3", num_sms=152)
    monkeypatch.setenv("TG_HOST_BLOCKS", "1024,1024,1536,4")
    h = tg.host_blocks(4100, 3000, 1500, path="tf32x3", num_sms=152)
    assert (h["row_blocks"], h["col_blocks"], h["first_block_rows"], h["block_rows"], h["block_cols"],
            h["split_row_blocks"], h["defer_copies_out"]) == (5, 2, 1024, 1024, 1536, 4, 0)
    assert h["model_ms"] > 0
    monkeypatch.setenv("TG_HOST_BLOCKS", "1024,1024,1536,4,1")
    assert tg.host_blocks(4100, 3000, 1500, path="tf32x3", num_sms=152)["defer_copies_out"] == 1
    for bad in ("1000,1024,1536,1", "1024,1024,1500,1", "1024,1024,1536,6", "128,128,256,1", "x"):
        monkeypatch.setenv("TG_HOST_BLOCKS", bad)
        assert tg.host_blocks(4100, 3000, 1500, path="tf32x3", num_sms=152) == model


def test_host_device_bytes_cover_every_product(monkeypatch):
    """The host call's workspace is sized over every product.  In this layout
    the middle row blocks are full width (1024 x 3000, a stream-K tail of 48
    pair units over 76 lanes with two partial slots per lane) while the first
    two and the last are not: their shapes alone would under-size it."""
    monkeypatch.setenv("TG_HOST_BLOCKS", "1024,1024,1536,2,1")
    got = tg.host_device_bytes(4100, 3000, 1500, path="tf32x3", num_sms=152)
    mid = tg.plan(1024, 3000, 1500, num_sms=152, path="tf32x3")
    assert mid["tail_lanes"] > 0 and mid["tail_kx"] == 0
    tail_slots = 2 * mid["tail_lanes"] * mid["pair"] * 128 * 256 * 4
    assert got["product_workspace"] >= tail_slots
    for shape in ((1024, 1536), (1024, 1464), (4, 3000)):
        q = tg.plan(*shape, 1500, num_sms=152, path="tf32x3")
        assert tail_slots > (2 * q["tail_lanes"] * q["pair"] * 128 * 256 * 4 if q["tail_kx"] == 0 else 0)
    # copies of A, B, C with 16-byte row pitches come on top
    assert got["total"] > got["product_workspace"] + 4 * (4100 * 1500 + 1500 * 3000 + 4100 * 3000)
    assert tg.host_device_bytes(0, 5, 5, num_sms=152) == {"total": 0, "product_workspace": 0}
    total = ctypes.c_size_t()
    assert tg.lib().tg_sgemm_host_device_bytes(-1, 4, 4, 0, 0, 152, ctypes.byref(total), None) == 1
    assert tg.lib().tg_sgemm_host_device_bytes(4, 4, 4, 0, 0, 152, None, None) == 1


def test_host_blocks_full_width_later_rows():
    """For 8192^3 the model cuts only the first row block into column blocks
    (the first product starts early) and computes the later row blocks full
    width, ending with a short row block (little work after the last copy in)."""
    h = tg.host_blocks(8192, 8192, 8192, path="tf32x3", num_sms=152)
    assert h["split_row_blocks"] == 1 and h["col_blocks"] > 1
    last = 8192 - h["first_block_rows"] - (h["row_blocks"] - 2) * h["block_rows"]
    assert 0 < last <= h["block_rows"]


def test_host_blocks_pipeline_large_products():
    """A large product is cut so that the first block's operands are a small
    part of A and B, and the modelled time beats a single block."""
    h = tg.host_blocks(8192, 8192, 8192, path="tf32x3", num_sms=152)
    assert h["row_blocks"] * h["col_blocks"] >= 4
    assert 4 * 8192 * (h["first_block_rows"] + h["block_cols"]) <= 0.5 * 4 * 8192 * 16384
    info = tg.binding.HostBlocksInfo()
    assert tg.lib().tg_sgemm_host_blocks(-1, 4, 4, 0, 152, ctypes.byref(info)) == 1
    assert tg.lib().tg_sgemm_host_blocks(4, 4, 4, 0, 152, None) == 1
    assert tg.lib().tg_sgemm_host_blocks(4, 4, 4, 7, 152, ctypes.byref(info)) == 1
    # below 2^33 multiply-adds: one block (bit-identical to the device entry)
    small = tg.host_blocks(777, 1029, 513, path="tf32x3", num_sms=152)
    assert (small["row_blocks"], small["col_blocks"]) == (1, 1)


def test_host_model_queued_copies_out(monkeypatch):
    """The host-pipeline model charges the ~40 us of a copy out only when it
    does not start right behind another queued copy out: with the copies out
    held until the copies in are done (they then queue), a layout with eight
    first-row-block products costs little more than one with four, and the
    model's choice for 8192^3 is the measured best of 80 layouts (first block
    2560 rows in 1024-column blocks, later blocks of 1024 rows, copies out
    held)."""
    monkeypatch.delenv("TG_HOST_BLOCKS", raising=False)
    h = tg.host_blocks(8192, 8192, 8192, path="tf32x3", num_sms=152)
    assert (h["first_block_rows"], h["block_rows"], h["block_cols"], h["defer_copies_out"]) == (2560, 1024, 1024, 1)

    def modelled(layout):
        monkeypatch.setenv("TG_HOST_BLOCKS", layout)
        return tg.host_blocks(8192, 8192, 8192, path="tf32x3", num_sms=152)["model_ms"]

    held8, held4 = modelled("2560,1024,1024,1,1"), modelled("2560,1024,2048,1,1")
    open8 = modelled("2560,1024,1024,1,0")
    # measured: 4.26, 4.41 and 4.50 ms
    assert held8 < held4 and held8 < open8
    assert 4.0 < held8 < 4.6
