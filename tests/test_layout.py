"""Host model of shared-memory banks for the access patterns the kernels use.

Bank model ("03 CUDA Shared Memory: Tiling, Bank Conflicts, and Reduction",
section "Bank Conflict"): 32 banks of 4-byte words; lanes hitting different
words of one bank are serialised; lanes reading the same word share it
(broadcast).  For 16-byte accesses a warp's request is served in 128-byte
wavefronts: the cost is the largest number of distinct 16-byte words that fall
on the same group of four banks.

Each test restates, from the kernel source, the address a lane uses and checks
that the pattern needs the minimum number of wavefronts.
"""
from math import gcd

import pytest


def wavefronts_32(addrs):
    """Serialisation degree of one warp-wide 4-byte access."""
    per_bank = {}
    for a in addrs:
        per_bank.setdefault((a // 4) % 32, set()).add(a // 4)
    return max(len(v) for v in per_bank.values())


def wavefronts_128(addrs):
    """Wavefronts of one warp-wide 16-byte access (addresses 16-byte aligned)."""
    words = {a // 16 for a in addrs}
    per_quad = {}
    for w in words:
        per_quad.setdefault(w % 8, set()).add(w)
    return max(len(v) for v in per_quad.values())


def min_wavefronts_128(addrs):
    return -(-len({a // 16 for a in addrs}) // 8)


# ------------------------------------------------------------- the pages' rules


@pytest.mark.parametrize("stride,degree", [(1, 1), (2, 2), (4, 4), (32, 32), (33, 1)])
def test_stride_conflict_degree_is_gcd(stride, degree):
    """Lane i reads word i*S: degree gcd(S, 32) (stride 2 is 2-way, 33 is free)."""
    assert wavefronts_32([4 * stride * lane for lane in range(32)]) == degree == gcd(stride, 32)


def test_transpose_padding():
    """tile[32][32] read down a column is 32-way; tile[32][33] is conflict-free."""
    col = 5
    assert wavefronts_32([4 * (r * 32 + col) for r in range(32)]) == 32
    assert wavefronts_32([4 * (r * 33 + col) for r in range(32)]) == 1


def test_xor_swizzle_rows_and_columns():
    """tile[r][c ^ r]: both a row and a column read touch all 32 banks once."""
    def addr(r, c):
        return 4 * (r * 32 + (c ^ r))
    for r in range(32):
        assert wavefronts_32([addr(r, c) for c in range(32)]) == 1
    for c in range(32):
        assert wavefronts_32([addr(r, c) for r in range(32)]) == 1


# ------------------------------------------------------------ FFMA kernel reads

BK = 32        # floats per A tile row (128 bytes, 128-byte TMA swizzle)
BN = 256       # floats per B tile row (no swizzle)


def ffma_a_addr(mw, lane, i, kk):
    """A fragment: float4 of row wm*32 + lm + 4i at 16-byte chunk kk/4,
    stored at chunk (kk/4) ^ (row % 8) (the 128-byte TMA swizzle)."""
    wm, lm = mw & 3, lane & 3
    r = wm * 32 + lm + 4 * i
    return r * BK * 4 + (((kk >> 2) ^ (r & 7)) * 16)


def ffma_b_addr(mw, lane, j, k):
    wn, ln = mw >> 2, lane >> 2
    return (k * BN + wn * 128 + 32 * j + 4 * ln) * 4


@pytest.mark.parametrize("mw", range(8))
def test_ffma_a_fragment_reads_conflict_free(mw):
    for i in range(8):
        for kk in range(0, BK, 4):
            addrs = [ffma_a_addr(mw, lane, i, kk) for lane in range(32)]
            assert wavefronts_128(addrs) == min_wavefronts_128(addrs) == 1


@pytest.mark.parametrize("mw", range(8))
def test_ffma_b_fragment_reads_conflict_free(mw):
    for j in range(4):
        for k in range(BK):
            addrs = [ffma_b_addr(mw, lane, j, k) for lane in range(32)]
            assert wavefronts_128(addrs) == min_wavefronts_128(addrs) == 1


def test_unswizzled_a_would_conflict():
    """Without the swizzle, the 4 rows read together (8 rows apart in a naive
    mapping, or 1 row apart at a 128-byte pitch) share a bank group."""
    addrs = [(lm + 4 * 0) * BK * 4 + 0 for lm in range(4) for _ in range(8)]
    assert wavefronts_128(addrs) == 4


# -------------------------------------------------------- pre-pass transpose


def test_prepass_transpose_tile_banks():
    """The pre-pass stages a 64 x 64 tile as tile[ty + 4j][tx] (row writes,
    tx = 0..63, a warp holds 32 consecutive tx; conflict-free with the
    65-float pitch) and reads it back one 16-byte destination group per
    thread: thread g = threadIdx + 256q reads tile[cl + e][rl], e = 0..3, with
    rl = g / 16 and cl = 4 (g % 16).  Those reads are two-way: lanes whose
    groups are 8 apart (cl 32 apart) land on the same bank."""
    pitch = 65
    for ty in range(4):
        for half in (0, 32):
            for j in range(16):
                writes = [4 * ((ty + 4 * j) * pitch + tx) for tx in range(half, half + 32)]
                assert wavefronts_32(writes) == 1
    for warp in range(8):
        for q in range(4):
            for e in range(4):
                reads = []
                for lane in range(32):
                    g = 32 * warp + lane + 256 * q
                    rl, cl = g >> 4, (g & 15) * 4
                    reads.append(4 * ((cl + e) * pitch + rl))
                assert wavefronts_32(reads) == 2


def split_tile_offset(pitch, r, c):
    """dst_offset of the split pre-pass modes (csrc/tg_kernels.cu), in floats:
    16 KiB tiles [r / 128][c / 16], row r % 128 of 32 floats, 16-byte group
    (c % 16) / 4 at position group ^ (r % 8)."""
    return ((r >> 7) * (pitch >> 4) + (c >> 4)) * 4096 + (r & 127) * 32 + ((((c & 15) >> 2) ^ (r & 7)) << 2) + (c & 3)


def bf16_run_offset(o, first):
    """bf16_offset of the tf32 + bf16 mode: the 8-byte run of the group at o
    inside logical group first (4: bf16 hi, 6: bf16 lo), in floats."""
    key = (o >> 5) & 7
    j = ((o >> 2) & 7) ^ key
    return (o & ~31) + (((first + (j >> 1)) ^ key) << 2) + ((j & 1) << 1)


@pytest.mark.parametrize("rows,pitch", [(300, 64), (128, 16), (1, 32)])
def test_split_tile_layouts_cover_each_slot_once(rows, pitch):
    """Both split layouts write every byte of the padded tiles exactly once:
    3xTF32 (hi at o, lo at o ^ 16) and tf32 + bf16 (tf32 hi at o, bf16 hi and
    lo in groups 4-7), and in the mixed layout the bf16 values of K 0-7 / 8-15
    of a row fill logical groups 4 / 5 (hi) and 6 / 7 (lo) in K order, so
    that one 32-byte MMA slice starts at group 4 or 6."""
    padded = -(-rows // 128) * 128
    total = padded // 128 * (pitch // 16) * 4096 * 4  # bytes
    tf32 = [0] * total
    mixed = [0] * total
    for r in range(padded):
        for c in range(pitch):
            o = split_tile_offset(pitch, r, c)
            for b in range(4):
                tf32[4 * o + b] += 1
                tf32[4 * (o ^ 16) + b] += 1
                mixed[4 * o + b] += 1
            for first in (4, 6):
                ob = 2 * bf16_run_offset(o, first) + (c & 3)  # in 2-byte units
                mixed[2 * ob] += 1
                mixed[2 * ob + 1] += 1
                # logical position inside the row: group first + (c % 16) / 8, slot (c % 8)
                row_base = o & ~31
                phys_group = ((ob // 2) - row_base) // 4
                logical = phys_group ^ (r & 7)
                assert logical == first + ((c & 15) >> 3)
                assert (ob - 2 * (row_base + 4 * phys_group)) == (c & 7)
    assert all(v == 1 for v in tf32)
    assert all(v == 1 for v in mixed)


def split_tile_h_offset(pitch, r, c):
    """dst_offset of the kSplitTf32H pre-pass mode, in floats: 16 KiB tiles
    [r / 128][c / 16]; hi in the first 8 KiB as rows of 16 floats, 16-byte
    group (c % 16) / 4 at position group ^ ((r / 2) % 4); lo 2048 floats on."""
    return ((r >> 7) * (pitch >> 4) + (c >> 4)) * 4096 + (r & 127) * 16 + \
        ((((c & 15) >> 2) ^ ((r >> 1) & 3)) << 2) + (c & 3)


def tma_swizzle_64(addr):
    """Where a 64-byte-swizzled TMA copy puts the byte at logical offset addr
    of its box (rows of 64 bytes, 512-byte aligned base): the 16-byte chunk
    index (address bits 4-5) is XORed with bits 7-8."""
    return addr ^ (((addr >> 7) & 3) << 4)


@pytest.mark.parametrize("rows,pitch", [(300, 64), (128, 16)])
def test_split_tile_h_matches_raw_tma_layout(rows, pitch):
    """The fused kernel reads pre-split operands and raw TMA tiles with the
    same descriptors, so the kSplitTf32H hi half must sit exactly where a
    64-byte-swizzled TMA box of the same 128 x 16 block puts the raw values,
    and hi + lo must cover each byte of the padded tiles once."""
    padded = -(-rows // 128) * 128
    total = padded // 128 * (pitch // 16) * 4096
    seen = [0] * total
    for r in range(padded):
        for c in range(pitch):
            o = split_tile_h_offset(pitch, r, c)
            tile = ((r >> 7) * (pitch >> 4) + (c >> 4)) * 4096
            assert 4 * (o - tile) == tma_swizzle_64(64 * (r & 127) + 4 * (c & 15))
            seen[o] += 1
            seen[o + 2048] += 1
    assert all(v == 1 for v in seen)


def bf16h_prepass_offset(pitch, r, c, part):
    """Where the kSplitBf16H pre-pass mode puts the bf16 value of (r, c)
    (part 0: bf16(hi), 1: bf16(lo)), in bytes: from the hi group's float
    offset o it recovers the row and the group, then writes 8-byte runs into
    the tile's second 8 KiB."""
    o = split_tile_h_offset(pitch, r, c & ~3)
    tile = o & ~4095
    row = (o >> 4) & 127
    key = (row >> 1) & 3
    g = ((o >> 2) & 3) ^ key
    base = tile + 2048 + 16 * row + 2 * (g & 1)        # floats
    run = base + 4 * (((2 * part) + (g >> 1)) ^ key)   # floats
    return 4 * run + 2 * (c & 3)


def bf16h_split_warp_offset(r, c, part):
    """Where the fused kernel's split warps put bf16 value (r, c) of a raw A
    tile (r < 128, c < 16), in bytes from the tile's second 8 KiB, starting
    from the raw 16-byte group that holds it (the 64-byte-swizzled TMA box)."""
    raw_byte = tma_swizzle_64(64 * r + 4 * (c & ~3))
    i = raw_byte // 16                  # the raw group's index, as the warps see it
    rr, key = i >> 2, ((i >> 2) >> 1) & 3
    g = (i & 3) ^ key
    assert rr == r and g == c // 4
    at = 64 * rr + 8 * (g & 1)
    return at + 16 * (((2 * part) + (g >> 1)) ^ key) + 2 * (c & 3)


def test_bf16h_layouts_agree_and_cover():
    """The tf32 + bf16 variant with a raw A reads A's bf16 tile (written by the
    split warps) and B's (written by the pre-pass) with one descriptor form,
    so both must put bf16 value (r, c) at the same place: K 0-7 / 8-15 of
    bf16(hi) in logical 16-byte groups 0 / 1 and bf16(lo) in 2 / 3, group j
    of row r at position j ^ ((r / 2) % 4), and every byte written once."""
    seen = [0] * 8192
    for r in range(128):
        for c in range(16):
            for part in (0, 1):
                pre = bf16h_prepass_offset(16, r, c, part) - 4 * 2048
                warp = bf16h_split_warp_offset(r, c, part)
                assert pre == warp, (r, c, part)
                logical = ((warp - 64 * r) // 16) ^ ((r >> 1) & 3)
                assert logical == 2 * part + (c >> 3) and (warp % 16) // 2 == c % 8
                seen[warp] += 1
                seen[warp + 1] += 1
    assert all(v == 1 for v in seen)


def test_bf16_split_warps_conflict_free():
    """The tf32 + bf16 split warps (split_raw_tile_bf16): thread t = 32w + l
    takes, in round u, row 8(w + 2u) + rig of its 8-row group, rig = {0, 1,
    4, 5} for lanes 0-15 and {2, 3, 6, 7} for lanes 16-31, four lanes per row
    at 16-byte position l % 4.  Every raw group is read once per stage; each
    quarter-warp's 16-byte loads hit 8 different bank groups and each
    half-warp's 8-byte stores (bf16 hi and bf16 lo) fill all 16 eight-byte
    slots of a bank row.  Four consecutive rows per half-warp would not."""
    def rig(lane):
        q = lane & 15
        return ((lane >> 4) << 1) + ((q >> 3) << 2) + ((q >> 2) & 1)

    def slots(rows_pos, part):
        out = []
        for r, p in rows_pos:
            key = (r >> 1) & 3
            c = p ^ key
            out.append(((64 * r + 16 * ((2 * part + (c >> 1)) ^ key) + 8 * (c & 1)) // 8) % 16)
        return out

    seen = set()
    for w in (0, 1):
        for u in range(8):
            lanes = [(8 * (w + 2 * u) + rig(l), l & 3) for l in range(32)]
            seen.update(lanes)
            for qw in range(4):
                assert len({(4 * r + p) % 8 for r, p in lanes[8 * qw:8 * qw + 8]}) == 8
            for hw in range(2):
                for part in (0, 1):
                    assert len(set(slots(lanes[16 * hw:16 * hw + 16], part))) == 16
    assert len(seen) == 512
    consecutive = [(r, p) for r in range(4) for p in range(4)]
    assert len(set(slots(consecutive, 0))) < 16


def test_fused_split_warps_access_conflict_free():
    """The split warps of the fused kernel move a raw 8 KiB tile to its lo
    half as 512 16-byte groups, thread t (0..63) taking t + 64u: each warp
    access covers 512 contiguous bytes, the minimum four wavefronts."""
    for u in range(8):
        for warp in range(2):
            addrs = [16 * (32 * warp + lane + 64 * u) for lane in range(32)]
            assert wavefronts_128(addrs) == min_wavefronts_128(addrs) == 4



def test_tensor_epilogue_staging_block_conflict_free():
    """The 3xTF32 epilogue's 32 x 32 staging block: lane r writes row r's
    eight 16-byte groups, group g at position g ^ (r % 8); it is read back
    either one column per lane (4-byte reads, one 128-byte row per store) or,
    in the 16-byte store form, lanes 8k..8k+7 reading the 8 groups of row k +
    4i.  Every access takes the minimum number of wavefronts."""
    def at(r, g):
        return 4 * (32 * r + 4 * (g ^ (r & 7)))  # bytes
    for g in range(8):  # the writes: lane r, group g (one instruction per g)
        addrs = [at(r, g) for r in range(32)]
        assert wavefronts_128(addrs) == min_wavefronts_128(addrs) == 4
    for r in range(32):  # 4-byte reads: lane l, column l of row r
        assert wavefronts_32([4 * (32 * r) + 4 * (l ^ ((r & 7) << 2)) for l in range(32)]) == 1
    for i in range(8):  # 16-byte reads: lane l, group l % 8 of row l // 8 + 4i
        addrs = [at(l // 8 + 4 * i, l % 8) for l in range(32)]
        assert wavefronts_128(addrs) == min_wavefronts_128(addrs) == 4


# ------------------------------------------------------- transpose workload


def transpose_tile_index(variant, r, c):
    """tile_index of csrc/tg_transpose.cu, in floats."""
    if variant == "padded":
        return r * 33 + c
    if variant == "swizzled":
        return r * 32 + (c ^ r)
    return r * 32 + c


@pytest.mark.parametrize("variant,read_degree", [("tile32", 32), ("padded", 1), ("swizzled", 1)])
def test_transpose_variants_bank_degrees(variant, read_degree):
    """Row writes into the tile are conflict-free for all three layouts; the
    column read (lane = tile row) is 32-way for tile[32][32] and free for the
    padded and swizzled layouts."""
    for ty in range(4):
        for j in range(8):
            writes = [4 * transpose_tile_index(variant, ty + 4 * j, tx) for tx in range(32)]
            reads = [4 * transpose_tile_index(variant, tx, ty + 4 * j) for tx in range(32)]
            assert wavefronts_32(writes) == 1
            assert wavefronts_32(reads) == read_degree

