"""Pins for the CPU oracle, none of which compares it with itself.

The oracle computes C[i][j] = sum_k A[i][k] B[k][j] in double, k ascending,
rounded once to float ("03 CUDA Shared Memory: Tiling, Bank Conflicts, and
Reduction", section "Shared Memory와 Tiling"; PMPP ch. 5 notes §5.5 for the
ghost zeros).  Each pin below checks it against something fixed by the
mathematics or worked by hand:

* hand-worked products in tests/golden/ (2x2, 3x3, rectangular, and the
  accumulation/rounding cases);
* identity and permutation matrices (exact);
* the transpose law oracle(B^T, A^T) = oracle(A, B)^T, bit for bit;
* brute force with exact rational arithmetic on tiny inputs;
* closed forms (all-ones, rank one);
* zero-padding (ghost element) invariance;
* exact integer products against int64 matrix multiplication;
* a float64 library product (within one ulp);
* strided operands, K = 0, empty shapes, rejected shapes;
* the sampled-row entry point against the same pins.

``test_mutants_are_caught`` plants plausible mistakes in copies of the oracle
source and checks that every one of them fails at least one pin.
"""
from __future__ import annotations

import os
import random
from fractions import Fraction

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# ---------------------------------------------------------------- helpers


def read_golden(name, tags=("A", "B", "C")):
    mats = {}
    with open(os.path.join(GOLDEN, name)) as f:
        lines = [ln.strip() for ln in f if ln.strip() and not ln.lstrip().startswith("#")]
    i = 0
    while i < len(lines):
        tag, r, c = lines[i].split()
        r, c = int(r), int(c)
        rows = [[float(v) for v in lines[i + 1 + k].split()] for k in range(r)]
        mats[tag] = np.array(rows, dtype=np.float32).reshape(r, c)
        i += 1 + r
    return tuple(mats[t] for t in tags)


def bits(x):
    return np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)


def assert_bitexact(got, want, what=""):
    g, w = bits(got), bits(want)
    bad = np.argwhere(g != w)
    assert bad.size == 0, f"{what}: {len(bad)} mismatches, first at {tuple(bad[0])}: {got[tuple(bad[0])]!r} vs {want[tuple(bad[0])]!r}"


def f32_to_fraction(x):
    return Fraction(float(np.float32(x)))


def round_fraction_to_f32(q: Fraction) -> np.float32:
    """Correctly rounded (nearest, ties to even) float32 of an exact rational."""
    if q == 0:
        return np.float32(0.0)
    f = np.float32(float(q))  # within one float32 ulp of the answer
    cands = {np.nextafter(f, np.float32(-np.inf)), f, np.nextafter(f, np.float32(np.inf))}
    best = None
    for c in cands:
        d = abs(Fraction(float(c)) - q)
        key = (d, int(np.array(c, dtype=np.float32).view(np.uint32)) & 1)
        if best is None or key < best[0]:
            best = (key, c)
    return np.float32(best[1])


def exact_product(A, B):
    M, K = A.shape
    N = B.shape[1]
    Af = [[f32_to_fraction(A[i, k]) for k in range(K)] for i in range(M)]
    Bf = [[f32_to_fraction(B[k, j]) for j in range(N)] for k in range(K)]
    return [[sum((Af[i][k] * Bf[k][j] for k in range(K)), Fraction(0)) for j in range(N)] for i in range(M)]


def ulp_distance(a, b):
    """Distance in float32 ulps (both finite)."""
    def key(x):
        u = np.array(x, dtype=np.float32).view(np.int32).astype(np.int64)
        return np.where(u < 0, -(u & 0x7FFFFFFF), u)
    return np.abs(key(a) - key(b))


def rand_f32(rng, shape, lo=-1.0, hi=1.0):
    return rng.uniform(lo, hi, size=shape).astype(np.float32)


# ------------------------------------------------------------------ pins
# Each pin takes the ctypes library so the mutation test can run it against
# a planted-mistake build.


def pin_hand_worked(lib):
    for name in ("hand_2x2.txt", "hand_3x3.txt", "hand_rect_1x3x2.txt", "hand_accumulation.txt"):
        A, B, C = read_golden(name)
        assert_bitexact(oracle.sgemm(A, B, lib=lib), C, name)


def pin_identity(lib):
    rng = np.random.default_rng(11)
    A = rand_f32(rng, (5, 7), -3, 3)
    assert_bitexact(oracle.sgemm(A, np.eye(7, dtype=np.float32), lib=lib), A, "A.I")
    assert_bitexact(oracle.sgemm(np.eye(5, dtype=np.float32), A, lib=lib), A, "I.A")


def pin_permutation(lib):
    rng = np.random.default_rng(12)
    B = rand_f32(rng, (6, 9))
    p = rng.permutation(6)
    P = np.eye(6, dtype=np.float32)[p]  # row i of P selects row p[i]
    assert_bitexact(oracle.sgemm(P, B, lib=lib), B[p], "P.B")
    A = rand_f32(rng, (4, 9))
    q = rng.permutation(9)
    Q = np.eye(9, dtype=np.float32)[:, q]  # column j of Q selects column q[j]
    assert_bitexact(oracle.sgemm(A, Q, lib=lib), A[:, q], "A.Q")


def pin_transpose_law(lib):
    rng = np.random.default_rng(13)
    for (M, N, K) in [(3, 5, 7), (17, 4, 33), (1, 9, 2), (8, 8, 1)]:
        A = rand_f32(rng, (M, K))
        B = rand_f32(rng, (K, N))
        C = oracle.sgemm(A, B, lib=lib)
        Ct = oracle.sgemm(np.ascontiguousarray(B.T), np.ascontiguousarray(A.T), lib=lib)
        assert_bitexact(Ct.T, C, f"transpose law {M}x{N}x{K}")


def pin_brute_force_exact(lib):
    """Inputs with few significant bits: every double partial sum is exact,
    so the oracle must equal the single correct rounding of the exact sum."""
    rng = random.Random(14)
    for _ in range(60):
        M, N, K = rng.randint(1, 5), rng.randint(1, 5), rng.randint(1, 6)

        def val():
            return rng.choice([-1, 1]) * rng.randint(0, 255) * 2.0 ** rng.randint(-6, 6)

        A = np.array([[val() for _ in range(K)] for _ in range(M)], dtype=np.float32)
        B = np.array([[val() for _ in range(N)] for _ in range(K)], dtype=np.float32)
        exact = exact_product(A, B)
        want = np.array([[round_fraction_to_f32(q) for q in row] for row in exact], dtype=np.float32)
        assert_bitexact(oracle.sgemm(A, B, lib=lib), want, f"exact brute force {M}x{N}x{K}")


def pin_brute_force_random(lib):
    """Full-precision random floats over a wide exponent range: the oracle is
    within one ulp of the correctly rounded exact sum (double rounding)."""
    rng = np.random.default_rng(15)
    total = off = 0
    for _ in range(40):
        M, N, K = (int(v) for v in rng.integers(1, 7, size=3))
        A = (rng.standard_normal((M, K)) * 2.0 ** rng.integers(-20, 20, size=(M, K))).astype(np.float32)
        B = (rng.standard_normal((K, N)) * 2.0 ** rng.integers(-20, 20, size=(K, N))).astype(np.float32)
        exact = exact_product(A, B)
        want = np.array([[round_fraction_to_f32(q) for q in row] for row in exact], dtype=np.float32)
        got = oracle.sgemm(A, B, lib=lib)
        d = ulp_distance(got, want)
        assert d.max() <= 1, f"brute force {M}x{N}x{K}: {d.max()} ulp"
        total += d.size
        off += int((d != 0).sum())
    assert off <= max(2, total // 100), f"{off} of {total} elements off by one ulp"


def pin_closed_forms(lib):
    for (M, N, K) in [(3, 4, 5), (7, 2, 300), (1, 1, 4097)]:
        C = oracle.sgemm(np.ones((M, K), np.float32), np.ones((K, N), np.float32), lib=lib)
        assert np.all(C == np.float32(K)), f"all-ones {M}x{N}x{K}"
    rng = np.random.default_rng(16)
    u = rng.integers(-5, 6, size=6).astype(np.float32)
    v = rng.integers(-5, 6, size=4).astype(np.float32)
    K = 37
    A = np.repeat(u[:, None], K, axis=1)  # A = u 1^T
    B = np.repeat(v[None, :], K, axis=0)  # B = 1 v^T
    C = oracle.sgemm(A, B, lib=lib)
    # the sum starts from +0.0, so a zero product row gives +0.0, never -0.0
    assert_bitexact(C, (K * np.outer(u, v)).astype(np.float32) + np.float32(0.0), "rank one")


def pin_zero_padding(lib):
    """Ghost elements: embedding in zeros leaves the valid block unchanged."""
    rng = np.random.default_rng(17)
    for (M, N, K) in [(5, 7, 9), (33, 65, 17), (1, 3, 1)]:
        A = rand_f32(rng, (M, K))
        B = rand_f32(rng, (K, N))
        Mp, Np, Kp = -(-M // 128) * 128, -(-N // 256) * 256, -(-K // 32) * 32
        Ap = np.zeros((Mp, Kp), np.float32)
        Ap[:M, :K] = A
        Bp = np.zeros((Kp, Np), np.float32)
        Bp[:K, :N] = B
        assert_bitexact(oracle.sgemm(Ap, Bp, lib=lib)[:M, :N], oracle.sgemm(A, B, lib=lib), "padding")
        # ... and the padded rows/columns of the product are exact zeros
        Cp = oracle.sgemm(Ap, Bp, lib=lib)
        assert np.all(bits(Cp[M:, :]) == 0) and np.all(bits(Cp[:, N:]) == 0)


def pin_integer_exact(lib):
    rng = np.random.default_rng(18)
    for (M, N, K) in [(16, 24, 40), (9, 5, 1000)]:
        Ai = rng.integers(-2, 3, size=(M, K))
        Bi = rng.integers(-2, 3, size=(K, N))
        want = (Ai.astype(np.int64) @ Bi.astype(np.int64)).astype(np.float32)
        assert_bitexact(oracle.sgemm(Ai.astype(np.float32), Bi.astype(np.float32), lib=lib), want, "integer")


def pin_float64_library(lib):
    rng = np.random.default_rng(19)
    A = rng.standard_normal((20, 300)).astype(np.float32)
    B = rng.standard_normal((300, 30)).astype(np.float32)
    want = (A.astype(np.float64) @ B.astype(np.float64)).astype(np.float32)
    assert ulp_distance(oracle.sgemm(A, B, lib=lib), want).max() <= 1


def pin_strides_and_edges(lib):
    rng = np.random.default_rng(20)
    M, N, K = 6, 5, 7
    Abig = rand_f32(rng, (M, K + 3))
    Bbig = rand_f32(rng, (K, N + 2))
    A, B = Abig[:, :K], Bbig[:, :N]
    Cbig = np.full((M, N + 4), np.nan, np.float32)
    oracle.sgemm(A, B, out=Cbig[:, :N], lib=lib)
    assert_bitexact(Cbig[:, :N], oracle.sgemm(np.ascontiguousarray(A), np.ascontiguousarray(B), lib=lib), "strided")
    assert np.all(np.isnan(Cbig[:, N:])), "columns beyond N were written"
    # hand value through strides: C[0][0] by its definition, exact rational
    q = sum((f32_to_fraction(A[0, k]) * f32_to_fraction(B[k, 0]) for k in range(K)), Fraction(0))
    assert ulp_distance(Cbig[0, 0], round_fraction_to_f32(q)) <= 1
    # K = 0: the empty sum is +0.0 everywhere
    C0 = np.full((3, 4), np.nan, np.float32)
    oracle.sgemm(np.zeros((3, 0), np.float32), np.zeros((0, 4), np.float32), out=C0, lib=lib)
    assert np.all(bits(C0) == 0)
    # M = 0 / N = 0 are no-ops
    assert oracle.sgemm(np.zeros((0, 3), np.float32), np.zeros((3, 2), np.float32), lib=lib).shape == (0, 2)
    assert oracle.sgemm(np.zeros((2, 3), np.float32), np.zeros((3, 0), np.float32), lib=lib).shape == (2, 0)


def pin_rows_entry(lib):
    A, B, C = read_golden("hand_3x3.txt")
    assert_bitexact(oracle.sgemm_rows(A, B, [2, 0], lib=lib), C[[2, 0]], "rows hand 3x3")
    rng = np.random.default_rng(21)
    A = rand_f32(rng, (40, 23))
    B = rand_f32(rng, (23, 19))
    rows = [39, 0, 17, 17, 5]
    exact = exact_product(A[rows], B)
    want = np.array([[round_fraction_to_f32(q) for q in row] for row in exact], dtype=np.float32)
    assert ulp_distance(oracle.sgemm_rows(A, B, rows, lib=lib), want).max() <= 1


# ------------------------------------------------- general form (op, alpha, beta)


def general(lib, op_a, op_b, alpha, A, B, beta, C0):
    C = np.array(C0, dtype=np.float32, copy=True)
    return oracle.sgemm_general(op_a, op_b, alpha, A, B, beta, C, lib=lib)


def pin_general_hand_worked(lib):
    A, B, C0, C = read_golden("hand_general_2x2.txt", ("A", "B", "C0", "C"))
    assert_bitexact(general(lib, 1, 0, 2.0, A, B, -0.5, C0), C, "hand general")


def pin_general_reduces_and_transposes(lib):
    """op N/N with alpha 1, beta 0 is the plain product; storing A or B
    transposed and flagging it gives the same bits; alpha = 2^e scales exactly."""
    rng = np.random.default_rng(31)
    for (M, N, K) in [(5, 7, 9), (17, 3, 40), (1, 1, 1)]:
        A = rand_f32(rng, (M, K))
        B = rand_f32(rng, (K, N))
        ref = oracle.sgemm(A, B, lib=lib)
        junk = np.full((M, N), np.nan, np.float32)
        assert_bitexact(general(lib, 0, 0, 1.0, A, B, 0.0, junk), ref, "N/N")
        At, Bt = np.ascontiguousarray(A.T), np.ascontiguousarray(B.T)
        assert_bitexact(general(lib, 1, 0, 1.0, At, B, 0.0, junk), ref, "T/N")
        assert_bitexact(general(lib, 0, 1, 1.0, A, Bt, 0.0, junk), ref, "N/T")
        assert_bitexact(general(lib, 1, 1, 1.0, At, Bt, 0.0, junk), ref, "T/T")
        assert_bitexact(general(lib, 0, 0, 4.0, A, B, 0.0, junk), 4 * ref, "alpha=4")
        assert_bitexact(general(lib, 1, 1, -0.25, At, Bt, 0.0, junk), -0.25 * ref, "alpha=-1/4")


def pin_general_alpha_beta_closed_forms(lib):
    rng = np.random.default_rng(32)
    M, N, K = 6, 5, 11
    A, B = rand_f32(rng, (M, K)), rand_f32(rng, (K, N))
    C0 = rand_f32(rng, (M, N), -3, 3)
    assert_bitexact(general(lib, 0, 0, 0.0, A, B, 1.0, C0), C0 + np.float32(0.0), "alpha=0 beta=1")
    assert_bitexact(general(lib, 0, 0, 0.0, A, B, -2.0, C0), -2 * C0 + np.float32(0.0), "alpha=0 beta=-2")
    # beta = 0 never reads C: NaN there has no effect
    assert_bitexact(general(lib, 0, 0, 1.0, A, B, 0.0, np.full((M, N), np.nan, np.float32)),
                    oracle.sgemm(A, B, lib=lib), "beta=0 ignores C")
    # K = 0: the empty sum, C = beta * C0
    assert_bitexact(general(lib, 0, 0, 3.0, np.zeros((M, 0), np.float32), np.zeros((0, N), np.float32),
                            0.5, C0), 0.5 * C0 + np.float32(0.0), "K=0")


def pin_general_brute_force_exact(lib):
    """Few-bit values: alpha*sum + beta*c is exact in double, so the oracle
    equals the single correct rounding of the exact rational result."""
    rng = random.Random(33)

    def val(lo=-6, hi=6):
        return rng.choice([-1, 1]) * rng.randint(0, 255) * 2.0 ** rng.randint(lo, hi)

    for _ in range(40):
        M, N, K = rng.randint(1, 4), rng.randint(1, 4), rng.randint(0, 5)
        op_a, op_b = rng.randint(0, 1), rng.randint(0, 1)
        alpha, beta = val(-3, 3), rng.choice([0.0, val(-3, 3)])
        A = np.array([[val() for _ in range(K)] for _ in range(M)], dtype=np.float32).reshape(M, K)
        B = np.array([[val() for _ in range(N)] for _ in range(K)], dtype=np.float32).reshape(K, N)
        C0 = np.array([[val() for _ in range(N)] for _ in range(M)], dtype=np.float32)
        exact = exact_product(A, B) if K > 0 else [[Fraction(0)] * N for _ in range(M)]
        want = np.array([[round_fraction_to_f32(Fraction(float(np.float32(alpha))) * exact[i][j]
                                                + Fraction(float(np.float32(beta))) * f32_to_fraction(C0[i, j]))
                          for j in range(N)] for i in range(M)], dtype=np.float32)
        As = np.ascontiguousarray(A.T) if op_a else A
        Bs = np.ascontiguousarray(B.T) if op_b else B
        got = general(lib, op_a, op_b, alpha, As.reshape(As.shape), Bs.reshape(Bs.shape), beta, C0)
        assert_bitexact(got + np.float32(0.0), want + np.float32(0.0), f"general brute force {M}x{N}x{K}")


# ------------------------------------------------------------------ transpose


def pin_transpose_hand_worked(lib):
    X, XT = read_golden("hand_transpose_2x3.txt", ("X", "XT"))
    assert_bitexact(oracle.transpose(X, lib=lib), XT, "hand transpose")


def pin_transpose_involution_and_library(lib):
    rng = np.random.default_rng(41)
    for (r, c) in [(1, 1), (1, 7), (33, 31), (64, 100)]:
        X = rand_f32(rng, (r, c), -5, 5)
        T = oracle.transpose(X, lib=lib)
        assert T.shape == (c, r)
        assert_bitexact(oracle.transpose(T, lib=lib), X, "transpose twice")
        assert_bitexact(T, np.ascontiguousarray(X.T), "numpy transpose")
        # element (r', c') of the result is X[c'][r'] (the definition)
        assert T[c - 1, 0] == X[0, c - 1] and T[0, r - 1] == X[r - 1, 0]
    # strided source (row pitch larger than the width)
    big = rand_f32(rng, (5, 9))
    assert_bitexact(oracle.transpose(big[:, :6], lib=lib), np.ascontiguousarray(big[:, :6].T), "strided")


# ---------------------------------------------------------------- reduction


def pin_sum_hand_worked_and_closed_forms(lib):
    # 1 + 2 + ... + 100 = 5050 (Gauss); 0.5 + 0.25 + 0.125 = 0.875
    assert oracle.reduce_sum(np.arange(1, 101, dtype=np.float32), lib=lib) == np.float32(5050)
    assert oracle.reduce_sum(np.array([0.5, 0.25, 0.125], np.float32), lib=lib) == np.float32(0.875)
    # the empty sum is +0.0; alternating +1/-1 cancels exactly
    z = oracle.reduce_sum(np.zeros(0, np.float32), lib=lib)
    assert z == 0 and not np.signbit(z)
    assert oracle.reduce_sum(np.tile(np.array([1.0, -1.0], np.float32), 500), lib=lib) == 0
    # a float accumulator would lose the small terms: 2^24 + 16 ones = 2^24 + 16
    x = np.concatenate([np.array([2.0 ** 24], np.float32), np.ones(16, np.float32)])
    assert oracle.reduce_sum(x, lib=lib) == np.float32(2 ** 24 + 16)


def pin_sum_exact_rational(lib):
    rng = np.random.default_rng(51)
    for n in (1, 2, 7, 50):
        x = (rng.standard_normal(n) * 2.0 ** rng.integers(-10, 10, size=n)).astype(np.float32)
        exact = sum((f32_to_fraction(v) for v in x), Fraction(0))
        want = round_fraction_to_f32(exact)
        assert ulp_distance(oracle.reduce_sum(x, lib=lib), want) <= 1, n
        ints = rng.integers(-2, 3, size=n).astype(np.float32)
        assert oracle.reduce_sum(ints, lib=lib) == np.float32(int(ints.astype(np.int64).sum()))


PINS = [pin_hand_worked, pin_identity, pin_permutation, pin_transpose_law, pin_brute_force_exact,
        pin_brute_force_random, pin_closed_forms, pin_zero_padding, pin_integer_exact,
        pin_float64_library, pin_strides_and_edges, pin_rows_entry, pin_general_hand_worked,
        pin_general_reduces_and_transposes, pin_general_alpha_beta_closed_forms,
        pin_general_brute_force_exact, pin_transpose_hand_worked, pin_transpose_involution_and_library,
        pin_sum_hand_worked_and_closed_forms, pin_sum_exact_rational]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin, oracle_lib):
    pin(oracle_lib)


def test_bad_shapes_rejected(oracle_lib):
    lib = oracle_lib
    buf = np.zeros(64, np.float32)
    p = buf.ctypes.data
    assert lib.tg_oracle_sgemm(-1, 2, 2, p, 2, p, 2, p, 2) == 1
    assert lib.tg_oracle_sgemm(2, 2, 3, p, 2, p, 2, p, 2) == 1  # lda < K
    assert lib.tg_oracle_sgemm(2, 3, 2, p, 2, p, 2, p, 3) == 1  # ldb < N
    assert lib.tg_oracle_sgemm(2, 3, 2, p, 2, p, 3, p, 2) == 1  # ldc < N
    rows = np.array([5], np.int64)
    assert lib.tg_oracle_sgemm_rows(1, rows.ctypes.data, 2, 2, 2, p, 2, p, 2, p, 2) == 1


def test_thread_count_does_not_change_results(oracle_lib):
    """Each output is one thread's ascending-k sum, so the result is the same
    bits whatever the number of OpenMP threads (the single-thread timing in
    the bench relies on this)."""
    rng = np.random.default_rng(11)
    A = rng.standard_normal((37, 300)).astype(np.float32)
    B = rng.standard_normal((300, 29)).astype(np.float32)
    n0 = oracle.threads(oracle_lib)
    try:
        many = oracle.sgemm(A, B, lib=oracle_lib)
        assert oracle.set_threads(1, oracle_lib) == 1
        one = oracle.sgemm(A, B, lib=oracle_lib)
    finally:
        oracle.set_threads(n0, oracle_lib)
    assert oracle.threads(oracle_lib) == n0
    assert np.array_equal(many.view(np.uint32), one.view(np.uint32))


def test_normal_inputs_statistics(oracle_lib):
    """RNG wiring: for i.i.d. N(0,1) operands each C element has mean 0 and
    variance K."""
    from shared_memory_tiled_fp32_gb300.workloads import make_inputs

    K = 1024
    A, B = make_inputs(64, 64, K, "normal", 99)
    C = oracle.sgemm(A.numpy(), B.numpy(), lib=oracle_lib).astype(np.float64)
    assert abs(C.mean()) < 5 * np.sqrt(K) / 64
    assert 0.85 < C.var() / K < 1.15


def test_workload_generators_are_seeded():
    from shared_memory_tiled_fp32_gb300.workloads import make_inputs

    a1, b1 = make_inputs(8, 9, 10, "int", 5)
    a2, b2 = make_inputs(8, 9, 10, "int", 5)
    assert bool((a1 == a2).all() and (b1 == b2).all())
    assert set(np.unique(a1.numpy())) <= {-2.0, -1.0, 0.0, 1.0, 2.0}
    u, _ = make_inputs(100, 1, 100, "uniform", 1)
    assert float(u.min()) >= -1.0 and float(u.max()) < 1.0


# -------------------------------------------------------------- mutants

MUTANTS = {
    "drop_last_term": ("for (int64_t k = 0; k < K; ++k)", "for (int64_t k = 0; k + 1 < K; ++k)"),
    "drop_first_term": ("for (int64_t k = 0; k < K; ++k)", "for (int64_t k = 1; k < K; ++k)"),
    "sign_flip": ("acc[j] += a * (double)B_row[j];", "acc[j] -= a * (double)B_row[j];"),
    "float_accumulator": ("acc[j] += a * (double)B_row[j];", "acc[j] = (float)(acc[j] + a * (double)B_row[j]);"),
    "ldb_for_lda": ("const float* B_row = B + k * ldb;", "const float* B_row = B + k * N;"),
    "c_row_stride": ("B, ldb, acc, C + i * ldc);", "B, ldb, acc, C + i * N);"),
    "transposed_A": ("const double a = (double)A_row[k];", "const double a = (double)A_row[k * 0] * (k + 1 > 0);"),
    "drop_last_column": ("for (int64_t j = 0; j < N; ++j) acc[j] += a", "for (int64_t j = 0; j + 1 < N; ++j) acc[j] += a"),
    "general_a_not_transposed": ("const double a = op_a ? (double)A[k * lda + i] : (double)A[i * lda + k];",
                                 "const double a = (double)A[i * lda + k];"),
    "general_b_not_transposed": ("const double b = op_b ? (double)B[j * ldb + k] : (double)B[k * ldb + j];",
                                 "const double b = (double)B[k * ldb + j];"),
    "general_alpha_dropped": ("double r = (double)alpha * s;", "double r = s;"),
    "general_beta_sign": ("if (beta != 0.0f) r += (double)beta", "if (beta != 0.0f) r -= (double)beta"),
    "general_reads_c_at_beta0": ("if (beta != 0.0f) r += (double)beta * (double)C[i * ldc + j];",
                                 "r += (double)beta * (double)C[i * ldc + j];"),
    "transpose_same_index": ("out[c * ld_out + r] = in[r * ld_in + c];", "out[r * ld_out + c] = in[r * ld_in + c];"),
    "transpose_drops_last_col": ("for (int64_t c = 0; c < cols; ++c) out[c * ld_out + r]",
                                 "for (int64_t c = 0; c + 1 < cols; ++c) out[c * ld_out + r]"),
    "sum_float_accumulator": ("for (int64_t i = 0; i < n; ++i) s += (double)x[i];",
                              "for (int64_t i = 0; i < n; ++i) s = (float)(s + (double)x[i]);"),
    "sum_skips_first": ("for (int64_t i = 0; i < n; ++i) s += (double)x[i];",
                        "for (int64_t i = 1; i < n; ++i) s += (double)x[i];"),
    "truncating_store": ("for (int64_t j = 0; j < N; ++j) C_row[j] = (float)acc[j];",
                         "for (int64_t j = 0; j < N; ++j) { float f = (float)acc[j]; if ((double)f - acc[j] > 0 && f > 0) f = nextafterf(f, 0.0f); else if ((double)f - acc[j] < 0 && f < 0) f = nextafterf(f, 0.0f); C_row[j] = f; }"),
}


_MUTANT_RUNNER = """
import sys
sys.path.insert(0, {tests!r}); sys.path.insert(0, {root!r})
import oracle, test_oracle
lib = oracle.load({so!r})
caught = []
for pin in test_oracle.PINS:
    try:
        pin(lib)
    except (AssertionError, RuntimeError, ValueError):
        caught.append(pin.__name__)
print("CAUGHT", ",".join(caught))
"""


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutants_are_caught(name, tmp_path):
    """Each planted mistake fails at least one pin.  The pins run in a child
    process: a mutant that writes out of bounds may crash it, which also
    counts as caught."""
    import subprocess
    import sys

    old, new = MUTANTS[name]
    with open(oracle._SRC) as f:
        src = f.read()
    assert old in src, f"mutation site for {name} not found"
    src = src.replace(old, new, 1)
    if "nextafterf" in new:
        src = "#include <math.h>\n" + src
    cpath = tmp_path / f"{name}.c"
    cpath.write_text(src)
    so = oracle.build(str(cpath), str(tmp_path / f"lib{name}.so"), extra_flags=["-lm"])
    tests_dir = os.path.dirname(os.path.abspath(__file__))
    code = _MUTANT_RUNNER.format(tests=tests_dir, root=os.path.dirname(tests_dir), so=so)
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300)
    if r.returncode != 0:
        return  # the mutant crashed the pins' process: caught
    line = [ln for ln in r.stdout.splitlines() if ln.startswith("CAUGHT")][-1]
    caught = [c for c in line[len("CAUGHT"):].strip().split(",") if c]
    assert caught, f"mutant {name} passed every pin"
