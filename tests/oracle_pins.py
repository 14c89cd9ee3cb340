"""Pins for the CPU oracle: checks that tie it to something other than itself.

Each pin takes an ``oracle.Oracle`` handle and raises AssertionError when the
oracle disagrees with

* brute force in exact rational arithmetic on tiny integer inputs,
* NumPy's float64 matmul on the decoded operands (a library routine),
* closed forms (ones, rank one, identity),
* the invariants (A*B)^T = B^T*A^T, SYRK = one triangle of GEMM(A, A^T),
  SYR2K = one triangle of GEMM(A, B^T) + GEMM(B, A^T), SYR2K(A, A) = 2 SYRK(A),
  SYR2K(A, B) = SYR2K(B, A),
  beta=1 accumulation = C0 + a beta=0 call, exact power-of-two alpha scaling,
* the BLAS conventions for alpha = 0, beta = 0 and k = 0,
* for the MXFP8 GEMM: exact rational brute force with power-of-two group
  scales, unit scales equal to the plain E4M3 GEMM, NumPy on the decoded
  operands, exact row and operand scaling,
* for the MXFP8 quantization (OCP MX conversion): every E4M3 code round trips,
  an exact rational restatement of the rule on random groups, ties to even,
  saturation, zero / NaN / infinite groups, short last groups and the rounding
  error bound.

``tests/test_oracle_mutants.py`` plants plausible mistakes in copies of the
oracle's C source and checks that every one of them fails at least one pin.
"""

from __future__ import annotations

from fractions import Fraction
import itertools

import numpy as np

import bm_inputs as gen

BF16_ONE = np.uint16(0x3F80)


def _stored(rows, cols, trans):
    """Stored shape of op(X) (rows x cols) for the trans flag."""
    return (cols, rows) if trans else (rows, cols)


def _int_bf16(shape, seed, lo=-4, hi=4, pad=0):
    vals = gen.integers(seed, shape[0] * shape[1], lo, hi).reshape(shape)
    bits = gen.f32_to_bf16_bits(vals)
    if pad:
        bits = gen.pad_ld(bits, shape[1] + pad, gen.BF16_NAN)
    return bits, vals


def _op(vals, trans):
    return vals.T if trans else vals


# --- brute force in exact arithmetic --------------------------------------------
def pin_gemm_bruteforce_exact(o):
    shapes = [(1, 1, 1), (3, 5, 4), (7, 2, 9), (4, 6, 1)]
    alphas = [Fraction(1), Fraction(-2), Fraction(1, 2)]
    betas = [Fraction(0), Fraction(1), Fraction(-1, 2)]
    seed = 100
    for (m, n, k), tA, tB in itertools.product(shapes, (0, 1), (0, 1)):
        seed += 3
        A, Av = _int_bf16(_stored(m, k, tA), seed, pad=3)
        B, Bv = _int_bf16(_stored(k, n, tB), seed + 1, pad=2)
        opA, opB = _op(Av, tA), _op(Bv, tB)
        prod = [[sum(Fraction(int(opA[i, p])) * Fraction(int(opB[p, j])) for p in range(k))
                 for j in range(n)] for i in range(m)]
        mag = [[sum(abs(int(opA[i, p]) * int(opB[p, j])) for p in range(k))
                for j in range(n)] for i in range(m)]
        for alpha, beta, cbf in itertools.product(alphas, betas, (False, True)):
            Cv = gen.integers(seed + 2, m * n, -8, 8).reshape(m, n)
            C = gen.f32_to_bf16_bits(Cv) if cbf else Cv.astype(np.float32)
            ref, bound = o.gemm(m, n, k, tA, tB, float(alpha), A, B, float(beta), C)
            for i in range(m):
                for j in range(n):
                    want = alpha * prod[i][j] + beta * Fraction(int(Cv[i, j]))
                    assert Fraction(ref[i, j]) == want, (m, n, k, tA, tB, alpha, beta, cbf, i, j)
                    assert bound[i, j] == mag[i][j], (m, n, k, tA, tB, i, j)


def pin_syrk_bruteforce_exact(o):
    for (n, k), uplo, trans in itertools.product([(1, 1), (5, 3), (6, 8)], (0, 1), (0, 1)):
        A, Av = _int_bf16(_stored(n, k, trans), 7 + n + 10 * k + 100 * uplo + 1000 * trans, pad=1)
        opA = _op(Av, trans)
        Cv = gen.integers(55, n * n, -8, 8).reshape(n, n)
        C = Cv.astype(np.float32)
        for alpha, beta in [(Fraction(1), Fraction(1)), (Fraction(-1, 2), Fraction(0)),
                            (Fraction(2), Fraction(-3, 2))]:
            ref, bound = o.syrk(uplo, trans, n, k, float(alpha), A, float(beta), C)
            for i in range(n):
                for j in range(n):
                    inside = (i >= j) if uplo == 0 else (i <= j)
                    if not inside:
                        assert np.isnan(ref[i, j]) and np.isnan(bound[i, j]), (n, k, uplo, trans, i, j)
                        continue
                    s = sum(Fraction(int(opA[i, p])) * Fraction(int(opA[j, p])) for p in range(k))
                    want = alpha * s + beta * Fraction(int(Cv[i, j]))
                    assert Fraction(ref[i, j]) == want, (n, k, uplo, trans, i, j)
                    assert bound[i, j] == sum(abs(int(opA[i, p]) * int(opA[j, p])) for p in range(k))


def pin_syr2k_bruteforce_exact(o):
    for (n, k), uplo, trans in itertools.product([(1, 1), (5, 3), (6, 7)], (0, 1), (0, 1)):
        A, Av = _int_bf16(_stored(n, k, trans), 300 + n + 10 * k + 100 * uplo + 1000 * trans, pad=2)
        B, Bv = _int_bf16(_stored(n, k, trans), 301 + n + 10 * k + 100 * uplo + 1000 * trans, pad=1)
        opA, opB = _op(Av, trans), _op(Bv, trans)
        Cv = gen.integers(57, n * n, -8, 8).reshape(n, n)
        for alpha, beta in [(Fraction(1), Fraction(0)), (Fraction(-1, 2), Fraction(1)), (Fraction(3), Fraction(-2))]:
            ref, bound = o.syr2k(uplo, trans, n, k, float(alpha), A, B, float(beta), Cv.astype(np.float32))
            for i in range(n):
                for j in range(n):
                    inside = (i >= j) if uplo == 0 else (i <= j)
                    if not inside:
                        assert np.isnan(ref[i, j]) and np.isnan(bound[i, j])
                        continue
                    s2 = sum(Fraction(int(opA[i, p])) * int(opB[j, p]) + Fraction(int(opB[i, p])) * int(opA[j, p])
                             for p in range(k))
                    assert Fraction(ref[i, j]) == alpha * s2 + beta * int(Cv[i, j]), (n, k, uplo, trans, i, j)
                    assert bound[i, j] == sum(abs(int(opA[i, p]) * int(opB[j, p])) + abs(int(opB[i, p]) * int(opA[j, p]))
                                              for p in range(k))


# --- NumPy float64 matmul ------------------------------------------------------
def pin_gemm_matches_numpy(o):
    m, n, k = 37, 29, 53
    for tA, tB in itertools.product((0, 1), (0, 1)):
        A = gen.matrix_bf16(*_stored(m, k, tA), "normal", seed=11 + tA)
        B = gen.matrix_bf16(*_stored(k, n, tB), "normal", seed=21 + tB)
        C = gen.matrix_f32(m, n, "normal", seed=31)
        a = _op(gen.bf16_bits_to_f32(A).astype(np.float64), tA)
        b = _op(gen.bf16_bits_to_f32(B).astype(np.float64), tB)
        alpha, beta = 0.75, -1.25
        want = alpha * (a @ b) + beta * C.astype(np.float64)
        ref, bound = o.gemm(m, n, k, tA, tB, alpha, A, B, beta, C)
        scale = abs(alpha) * (np.abs(a) @ np.abs(b)) + abs(beta) * np.abs(C)
        assert np.all(np.abs(ref - want) <= 1e-13 * scale + 1e-300), (tA, tB)
        assert np.allclose(bound, np.abs(a) @ np.abs(b), rtol=1e-13, atol=0), (tA, tB)


def pin_syrk_matches_numpy(o):
    n, k = 23, 31
    for uplo, trans in itertools.product((0, 1), (0, 1)):
        A = gen.matrix_bf16(*_stored(n, k, trans), "normal", seed=41 + trans)
        C = gen.symmetric_f32(n, seed=43)
        a = _op(gen.bf16_bits_to_f32(A).astype(np.float64), trans)
        want = 1.5 * (a @ a.T) + 0.5 * C.astype(np.float64)
        ref, _ = o.syrk(uplo, trans, n, k, 1.5, A, 0.5, C)
        mask = np.tril(np.ones((n, n), bool)) if uplo == 0 else np.triu(np.ones((n, n), bool))
        scale = 1.5 * (np.abs(a) @ np.abs(a).T) + 0.5 * np.abs(C)
        assert np.all(np.abs(ref[mask] - want[mask]) <= 1e-13 * scale[mask]), (uplo, trans)
        assert np.all(np.isnan(ref[~mask])), (uplo, trans)


def pin_syr2k_matches_numpy(o):
    n, k = 21, 33
    for uplo, trans in itertools.product((0, 1), (0, 1)):
        A = gen.matrix_bf16(*_stored(n, k, trans), "normal", seed=141 + trans)
        B = gen.matrix_bf16(*_stored(n, k, trans), "normal", seed=151 + trans)
        C = gen.symmetric_f32(n, seed=161)
        a = _op(gen.bf16_bits_to_f32(A).astype(np.float64), trans)
        b = _op(gen.bf16_bits_to_f32(B).astype(np.float64), trans)
        want = -0.5 * (a @ b.T + b @ a.T) + 2.0 * C.astype(np.float64)
        ref, bound = o.syr2k(uplo, trans, n, k, -0.5, A, B, 2.0, C)
        mask = np.tril(np.ones((n, n), bool)) if uplo == 0 else np.triu(np.ones((n, n), bool))
        mag = np.abs(a) @ np.abs(b).T + np.abs(b) @ np.abs(a).T
        assert np.all(np.abs(ref[mask] - want[mask]) <= 1e-13 * (0.5 * mag[mask] + 2.0 * np.abs(C[mask])))
        assert np.allclose(bound[mask], mag[mask], rtol=1e-13, atol=0)
        assert np.all(np.isnan(ref[~mask]))


# --- closed forms -----------------------------------------------------------------
def pin_identity(o):
    n = 19
    eye = np.zeros((n, n), np.uint16)
    eye[np.arange(n), np.arange(n)] = BF16_ONE
    B = gen.matrix_bf16(n, 13, "normal", seed=5)
    ref, _ = o.gemm(n, 13, n, 0, 0, 1.0, eye, B)
    assert np.array_equal(ref, gen.bf16_bits_to_f32(B).astype(np.float64))
    A = gen.matrix_bf16(11, n, "normal", seed=6)
    ref, _ = o.gemm(11, n, n, 0, 0, 1.0, A, eye)
    assert np.array_equal(ref, gen.bf16_bits_to_f32(A).astype(np.float64))


def pin_closed_forms(o):
    m, n, k = 9, 12, 40
    ones_a = np.full((m, k), BF16_ONE, np.uint16)
    ones_b = np.full((k, n), BF16_ONE, np.uint16)
    ref, bound = o.gemm(m, n, k, 0, 0, 1.0, ones_a, ones_b)
    assert np.all(ref == k) and np.all(bound == k)
    # rank one: op(A)[i][p] = i - 2, op(B)[p][j] = j - 1  ->  C = k (i - 2)(j - 1)
    x = np.arange(m, dtype=np.float64) - 2
    y = np.arange(n, dtype=np.float64) - 1
    A = gen.f32_to_bf16_bits(np.repeat(x[:, None], k, axis=1))
    B = gen.f32_to_bf16_bits(np.repeat(y[None, :], k, axis=0))
    ref, bound = o.gemm(m, n, k, 0, 0, -3.0, A, B)
    assert np.array_equal(ref, -3.0 * k * np.outer(x, y))
    assert np.array_equal(bound, k * np.abs(np.outer(x, y)))
    # SYRK of rows of constant value v_i: C = k v_i v_j
    v = np.arange(n, dtype=np.float64) - 5
    Asy = gen.f32_to_bf16_bits(np.repeat(v[:, None], k, axis=1))
    ref, _ = o.syrk(0, 0, n, k, 1.0, Asy)
    low = np.tril(np.ones((n, n), bool))
    assert np.array_equal(ref[low], (k * np.outer(v, v))[low])


# --- invariants ---------------------------------------------------------------------
def pin_transpose_identity(o):
    m, n, k = 21, 17, 26
    for tA, tB in itertools.product((0, 1), (0, 1)):
        A = gen.matrix_bf16(*_stored(m, k, tA), "normal", seed=61)
        B = gen.matrix_bf16(*_stored(k, n, tB), "normal", seed=62)
        c1, b1 = o.gemm(m, n, k, tA, tB, 1.0, A, B)
        c2, b2 = o.gemm(n, m, k, 1 - tB, 1 - tA, 1.0, B, A)
        assert np.array_equal(c1, c2.T) and np.array_equal(b1, b2.T), (tA, tB)


def pin_syrk_is_gemm_triangle(o):
    n, k = 27, 35
    low = np.tril(np.ones((n, n), bool))
    for trans in (0, 1):
        A = gen.matrix_bf16(*_stored(n, k, trans), "normal", seed=71)
        g, gb = o.gemm(n, n, k, trans, 1 - trans, 1.0, A, A)
        for uplo, mask in ((0, low), (1, low.T)):
            s, sb = o.syrk(uplo, trans, n, k, 1.0, A)
            assert np.array_equal(s[mask], g[mask]) and np.array_equal(sb[mask], gb[mask]), (uplo, trans)


def pin_syr2k_invariants(o):
    n, k = 19, 24
    low = np.tril(np.ones((n, n), bool))
    for trans in (0, 1):
        A = gen.matrix_bf16(*_stored(n, k, trans), "normal", seed=171)
        B = gen.matrix_bf16(*_stored(n, k, trans), "normal", seed=172)
        s2, b2 = o.syr2k(0, trans, n, k, 1.0, A, B)
        # one triangle of GEMM(A, B^T) + GEMM(B, A^T)
        g1, gb1 = o.gemm(n, n, k, trans, 1 - trans, 1.0, A, B)
        g2, gb2 = o.gemm(n, n, k, trans, 1 - trans, 1.0, B, A)
        assert np.array_equal(s2[low], (g1 + g2)[low]) and np.array_equal(b2[low], (gb1 + gb2)[low])
        # swapping the operands changes nothing
        t2, _ = o.syr2k(0, trans, n, k, 1.0, B, A)
        assert np.array_equal(s2[low], t2[low])
        # SYR2K(A, A) = 2 SYRK(A)
        d2, db = o.syr2k(1, trans, n, k, 0.75, A, A)
        sy, sb = o.syrk(1, trans, n, k, 0.75, A)
        up = low.T
        assert np.array_equal(d2[up], 2.0 * sy[up]) and np.array_equal(db[up], 2.0 * sb[up])


def pin_beta_accumulation(o):
    m, n, k = 14, 22, 18
    A, _ = _int_bf16((m, k), 81, -8, 8)
    B, _ = _int_bf16((k, n), 82, -8, 8)
    C0 = gen.integers(83, m * n, -100, 100).reshape(m, n).astype(np.float32)
    acc, _ = o.gemm(m, n, k, 0, 0, 1.0, A, B, 1.0, C0)
    plain, _ = o.gemm(m, n, k, 0, 0, 1.0, A, B)
    assert np.array_equal(acc, C0.astype(np.float64) + plain)
    C0b = gen.f32_to_bf16_bits(C0)
    acc_b, _ = o.gemm(m, n, k, 0, 0, 1.0, A, B, 1.0, C0b)
    assert np.array_equal(acc_b, gen.bf16_bits_to_f32(C0b).astype(np.float64) + plain)


def pin_alpha_scaling(o):
    m, n, k = 10, 8, 33
    A = gen.matrix_bf16(m, k, "normal", seed=91)
    B = gen.matrix_bf16(k, n, "normal", seed=92)
    one, b1 = o.gemm(m, n, k, 0, 0, 1.0, A, B)
    two, b2 = o.gemm(m, n, k, 0, 0, 2.0, A, B)
    neg, _ = o.gemm(m, n, k, 0, 0, -0.25, A, B)
    assert np.array_equal(two, 2.0 * one) and np.array_equal(neg, -0.25 * one)
    assert np.array_equal(b1, b2)


# --- BLAS conventions ---------------------------------------------------------------------
def pin_special_values(o):
    m, n, k = 6, 7, 5
    nanA = np.full((m, k), gen.BF16_NAN, np.uint16)
    nanB = np.full((k, n), gen.BF16_NAN, np.uint16)
    C = gen.matrix_f32(m, n, "normal", seed=101)
    ref, bound = o.gemm(m, n, k, 0, 0, 0.0, nanA, nanB, 2.0, C)      # alpha = 0: A, B unread
    assert np.array_equal(ref, 2.0 * C.astype(np.float64)) and np.all(bound == 0)
    A = gen.matrix_bf16(m, k, "normal", seed=102)
    B = gen.matrix_bf16(k, n, "normal", seed=103)
    nanC = np.full((m, n), np.nan, np.float32)
    ref, _ = o.gemm(m, n, k, 0, 0, 1.0, A, B, 0.0, nanC)              # beta = 0: C unread
    assert np.all(np.isfinite(ref))
    ref, bound = o.gemm(m, n, 0, 0, 0, 1.0, A, B, -1.0, C)            # k = 0: beta * C
    assert np.array_equal(ref, -C.astype(np.float64)) and np.all(bound == 0)
    s, _ = o.syrk(0, 0, m, k, 0.0, nanA, 1.0, C[:, :m].copy())
    assert np.array_equal(s[np.tril(np.ones((m, m), bool))],
                          C[:, :m].astype(np.float64)[np.tril(np.ones((m, m), bool))])


def pin_entries_agree(o):
    m, n, k = 33, 41, 27
    rng = np.random.default_rng(5)
    rows = rng.integers(0, m, 200)
    cols = rng.integers(0, n, 200)
    for tA, tB in itertools.product((0, 1), (0, 1)):
        A = gen.matrix_bf16(*_stored(m, k, tA), "normal", seed=111)
        B = gen.matrix_bf16(*_stored(k, n, tB), "normal", seed=112)
        C = gen.f32_to_bf16_bits(gen.matrix_f32(m, n, "normal", seed=113))
        full, fb = o.gemm(m, n, k, tA, tB, 0.5, A, B, 1.0, C)
        e, eb = o.gemm_entries(k, tA, tB, 0.5, A, B, rows, cols, 1.0, C)
        assert np.array_equal(e, full[rows, cols]) and np.array_equal(eb, fb[rows, cols])
    As = gen.matrix_bf16(m, k, "normal", seed=114)
    Cs = gen.symmetric_f32(m, seed=115)
    r2 = rng.integers(0, m, 200)
    for uplo in (0, 1):
        full, _ = o.syrk(uplo, 0, m, k, 1.0, As, 1.0, Cs)
        e, _ = o.syrk_entries(uplo, 0, k, 1.0, As, rows, r2, 1.0, Cs)
        assert np.array_equal(e, full[rows, r2], equal_nan=True)
        Bs = gen.matrix_bf16(m, k, "normal", seed=116)
        full2, fb2 = o.syr2k(uplo, 0, m, k, 0.5, As, Bs, 1.0, Cs)
        e2, eb2 = o.syr2k_entries(uplo, 0, k, 0.5, As, Bs, rows, r2, 1.0, Cs)
        assert np.array_equal(e2, full2[rows, r2], equal_nan=True)
        assert np.array_equal(eb2, fb2[rows, r2], equal_nan=True)


# --- FP8 E4M3 GEMM ---------------------------------------------------------------------
def _int_e4m3(shape, seed, lo=-8, hi=8, pad=0):
    vals = gen.integers(seed, shape[0] * shape[1], lo, hi).reshape(shape)
    codes = gen.f32_to_e4m3_bits(vals)
    if pad:
        codes = gen.pad_ld(codes, shape[1] + pad, np.uint8(0x7F))  # NaN padding, never read
    return codes, vals


def pin_e4m3_decode_every_code(o):
    # 1 x 1 x 1 products with B = 1.0 (code 0x38) decode each A code
    one = np.full((1, 1), 0x38, np.uint8)
    for c in range(256):
        ref, _ = o.gemm_e4m3(1, 1, 1, 1.0, np.full((1, 1), c, np.uint8), one)
        want = gen.e4m3_bits_to_f32(np.uint8([c]))[0]
        if np.isnan(want):
            assert np.isnan(ref[0, 0]), c
        else:
            assert ref[0, 0] == want, (hex(c), ref[0, 0], want)


def pin_e4m3_bruteforce_exact(o):
    for (m, n, k) in [(1, 1, 1), (3, 4, 5), (6, 2, 9)]:
        A, Av = _int_e4m3((m, k), 200 + m, pad=5)
        B, Bv = _int_e4m3((n, k), 201 + n, pad=3)
        Cv = gen.integers(202, m * n, -9, 9).reshape(m, n)
        for alpha, beta in [(Fraction(1), Fraction(0)), (Fraction(-1, 4), Fraction(2))]:
            ref, bound = o.gemm_e4m3(m, n, k, float(alpha), A, B, float(beta), Cv.astype(np.float32))
            for i in range(m):
                for j in range(n):
                    s2 = sum(int(Av[i, p]) * int(Bv[j, p]) for p in range(k))
                    assert Fraction(ref[i, j]) == alpha * s2 + beta * int(Cv[i, j]), (m, n, k, i, j)
                    assert bound[i, j] == sum(abs(int(Av[i, p]) * int(Bv[j, p])) for p in range(k))


def pin_e4m3_equals_bf16_gemm_on_same_values(o):
    # E4M3 values are exact in bf16: the FP8 GEMM must equal the (pinned) bf16 GEMM with op(B) = B^T
    m, n, k = 23, 19, 41
    A = gen.matrix_e4m3(m, k, "normal", seed=211, std=4.0)
    B = gen.matrix_e4m3(n, k, "normal", seed=212, std=0.5)
    Ab = gen.f32_to_bf16_bits(gen.e4m3_bits_to_f32(A))
    Bb = gen.f32_to_bf16_bits(gen.e4m3_bits_to_f32(B))
    C = gen.matrix_f32(m, n, "normal", seed=213)
    r8, b8 = o.gemm_e4m3(m, n, k, 0.5, A, B, -1.5, C)
    r16, b16 = o.gemm(m, n, k, 0, 1, 0.5, Ab, Bb, -1.5, C)
    assert np.array_equal(r8, r16) and np.array_equal(b8, b16)
    rows = np.arange(m) % m
    cols = (np.arange(m) * 7) % n
    e, eb = o.gemm_e4m3_entries(k, 0.5, A, B, rows, cols, -1.5, C)
    assert np.array_equal(e, r8[rows, cols]) and np.array_equal(eb, b8[rows, cols])


def pin_e4m3_matches_numpy(o):
    m, n, k = 31, 17, 64
    A = gen.matrix_e4m3(m, k, "normal", seed=221)
    B = gen.matrix_e4m3(n, k, "uniform", seed=222, lo=-2, hi=2)
    a = gen.e4m3_bits_to_f32(A).astype(np.float64)
    b = gen.e4m3_bits_to_f32(B).astype(np.float64)
    ref, bound = o.gemm_e4m3(m, n, k, 2.0, A, B)
    assert np.all(np.abs(ref - 2.0 * a @ b.T) <= 1e-13 * 2.0 * (np.abs(a) @ np.abs(b).T))
    assert np.allclose(bound, np.abs(a) @ np.abs(b).T, rtol=1e-13, atol=0)


# --- MXFP8: E4M3 data with one UE8M0 scale per group of 32 along K --------------------
def _ue8m0(rows, groups, seed, lo=124, hi=130, pad=0):
    codes = gen.integers(seed, rows * groups, lo, hi).reshape(rows, groups).astype(np.uint8)
    if pad:
        codes = gen.pad_ld(codes, groups + pad, np.uint8(0xFF))  # NaN scales: never read
    return codes


def _pow2(e):
    return Fraction(2) ** int(e)


def pin_mxfp8_bruteforce_exact(o):
    # k crosses group boundaries (33 = 32 + 1, 70 = 2 * 32 + 6, 96 = 3 whole groups)
    for (m, n, k) in [(1, 1, 1), (2, 3, 33), (3, 2, 70), (2, 2, 96)]:
        g = (k + 31) // 32
        A, Av = _int_e4m3((m, k), 300 + k, pad=4)
        B, Bv = _int_e4m3((n, k), 301 + k, pad=2)
        SA = _ue8m0(m, g, 302 + k, pad=2)
        SB = _ue8m0(n, g, 303 + k, pad=1)
        Cv = gen.integers(304 + k, m * n, -9, 9).reshape(m, n)
        for alpha, beta in [(Fraction(1), Fraction(0)), (Fraction(-1, 2), Fraction(3))]:
            ref, bound = o.gemm_mxfp8(m, n, k, float(alpha), A, SA, B, SB, float(beta), Cv.astype(np.float32))
            for i in range(m):
                for j in range(n):
                    terms = [int(Av[i, p]) * _pow2(int(SA[i, p // 32]) - 127) * int(Bv[j, p])
                             * _pow2(int(SB[j, p // 32]) - 127) for p in range(k)]
                    assert Fraction(ref[i, j]) == alpha * sum(terms) + beta * int(Cv[i, j]), (m, n, k, i, j)
                    assert Fraction(bound[i, j]) == sum(abs(t) for t in terms), (m, n, k, i, j)


def pin_mxfp8_unit_scales_equal_e4m3(o):
    # code 127 is 2^0: the block-scaled GEMM must reduce to the (pinned) plain E4M3 GEMM
    m, n, k = 13, 11, 100
    A = gen.matrix_e4m3(m, k, "normal", seed=311, std=2.0)
    B = gen.matrix_e4m3(n, k, "normal", seed=312)
    ones_a = np.full((m, 4), 127, np.uint8)
    ones_b = np.full((n, 4), 127, np.uint8)
    C = gen.matrix_f32(m, n, "normal", seed=313)
    r, b = o.gemm_mxfp8(m, n, k, 0.25, A, ones_a, B, ones_b, -2.0, C)
    r8, b8 = o.gemm_e4m3(m, n, k, 0.25, A, B, -2.0, C)
    assert np.array_equal(r, r8) and np.array_equal(b, b8)


def _mx_decode(codes, scales, k):
    vals = gen.e4m3_bits_to_f32(codes).astype(np.float64)[:, :k]
    per = np.repeat(np.ldexp(1.0, scales.astype(np.int64) - 127), 32, axis=1)[:, :k]
    return vals * per


def pin_mxfp8_matches_numpy(o):
    m, n, k = 21, 17, 200
    g = (k + 31) // 32
    A = gen.matrix_e4m3(m, k, "normal", seed=321)
    B = gen.matrix_e4m3(n, k, "uniform", seed=322, lo=-3, hi=3)
    SA = _ue8m0(m, g, 323, lo=110, hi=140)
    SB = _ue8m0(n, g, 324, lo=110, hi=140)
    a, b = _mx_decode(A, SA, k), _mx_decode(B, SB, k)
    ref, bound = o.gemm_mxfp8(m, n, k, 1.5, A, SA, B, SB)
    assert np.all(np.abs(ref - 1.5 * a @ b.T) <= 1e-13 * 1.5 * (np.abs(a) @ np.abs(b).T))
    assert np.allclose(bound, np.abs(a) @ np.abs(b).T, rtol=1e-13, atol=0)


def pin_mxfp8_scaling_exact(o):
    # raising every scale of row i of SA by d multiplies row i of the products by 2^d;
    # raising every code of SB by 1 doubles every product
    m, n, k = 9, 7, 96
    A = gen.matrix_e4m3(m, k, "normal", seed=331)
    B = gen.matrix_e4m3(n, k, "normal", seed=332)
    SA = _ue8m0(m, 3, 333)
    SB = _ue8m0(n, 3, 334)
    ref, bound = o.gemm_mxfp8(m, n, k, 1.0, A, SA, B, SB)
    SA2 = SA.copy()
    SA2[4] += 3
    r2, b2 = o.gemm_mxfp8(m, n, k, 1.0, A, SA2, B, SB)
    want = ref.copy()
    want[4] *= 8.0
    assert np.array_equal(r2, want)
    r3, _ = o.gemm_mxfp8(m, n, k, 1.0, A, SA, B, (SB + 1).astype(np.uint8))
    assert np.array_equal(r3, 2.0 * ref)
    rows = np.array([0, 4, 8, 3])
    cols = np.array([6, 0, 2, 3])
    e, eb = o.gemm_mxfp8_entries(k, 1.0, A, SA, B, SB, rows, cols)
    assert np.array_equal(e, ref[rows, cols]) and np.array_equal(eb, bound[rows, cols])


E4M3_FINITE = [c for c in range(256) if (c & 0x7F) != 0x7F]


def _e4m3_frac(c):
    e, m = (c >> 3) & 0xF, c & 7
    mag = Fraction(m, 8) * _pow2(-6) if e == 0 else (1 + Fraction(m, 8)) * _pow2(e - 7)
    return -mag if c & 0x80 else mag


def _floor_log2(x: Fraction) -> int:
    # largest e with 2^e <= x, for x > 0
    e = x.numerator.bit_length() - x.denominator.bit_length()
    while _pow2(e) > x:
        e -= 1
    while _pow2(e + 1) <= x:
        e += 1
    return e


def _mx_rule(group_vals):
    """The OCP MX conversion of one group, restated in exact rationals: (scale code, codes)."""
    fr = [Fraction(float(v)) for v in group_vals]
    amax = max((abs(v) for v in fr), default=Fraction(0))
    e = -127 if amax == 0 else max(-127, min(127, _floor_log2(amax) - 8))
    out = []
    for v in fr:
        y = v / _pow2(e)
        if abs(y) >= 448:
            c = 0x7E
        else:
            best = min(range(0x7F), key=lambda c: (abs(_e4m3_frac(c) - abs(y)), c & 1))
            c = best
        out.append(c | 0x80 if (y < 0 or (y == 0 and np.signbit(float(v)))) else c)
    return e + 127, out


def pin_quantize_every_code_round_trips(o):
    # a group led by 256 (= 2^8, scale 2^0) carries each finite E4M3 value through unchanged
    codes = np.array(E4M3_FINITE, dtype=np.uint8)
    vals = gen.e4m3_bits_to_f32(codes)
    rows = -(-len(vals) // 31)
    X = np.zeros((rows, 32), np.float32)
    X[:, 0] = 256.0
    flat = np.zeros(rows * 31, np.float32)
    flat[:len(vals)] = vals
    X[:, 1:] = flat.reshape(rows, 31)
    Q, S = o.quantize_mxfp8(gen.f32_to_bf16_bits(X))
    assert np.all(S == 127)
    assert np.all(Q[:, 0] == 0x78)
    got = Q[:, 1:].reshape(-1)[:len(vals)]
    want = codes.copy()
    want[want == 0x80] = 0x80  # -0 keeps its sign
    assert np.array_equal(got, want), np.nonzero(got != want)


def pin_quantize_matches_exact_rule(o):
    rng_rows, k = 6, 70  # groups of 32, 32 and 6
    X = gen.matrix_bf16(rng_rows, k, "normal", seed=341, std=3.0)
    X[1] = gen.f32_to_bf16_bits(gen.bf16_bits_to_f32(X[1]) * np.float32(2e-38))   # tiny: scale clamped at 2^-127
    X[2] = gen.f32_to_bf16_bits(gen.bf16_bits_to_f32(X[2]) * np.float32(1e20))     # large exponents
    Q, S = o.quantize_mxfp8(gen.pad_ld(X, k + 6, gen.BF16_NAN), k)
    vals = gen.bf16_bits_to_f32(X)
    assert np.all(S[1] == 0)  # floor(log2(amax)) - 8 < -127 in every group of row 1
    for i in range(rng_rows):
        for g in range(3):
            code, want = _mx_rule(vals[i, 32 * g:min(k, 32 * g + 32)])
            assert S[i, g] == code, (i, g, S[i, g], code)
            assert list(Q[i, 32 * g:min(k, 32 * g + 32)]) == want, (i, g)


def pin_quantize_ties_saturation_specials(o):
    X = np.zeros((5, 40), np.float32)
    # row 0: amax 256 (scale 2^0); E4M3 steps by 1 in [8, 16) and by 2 in [16, 32), so 8.5
    # (8|9), 9.5 (9|10) and 17 (16|18) are ties: the even mantissas give 8, 10 and 16
    X[0, :4] = [256.0, 8.5, 9.5, 17.0]
    X[0, 32:] = [-1.0, 0.0, 0.0, 0.0, 0.0, 0.0, 0.0, 2.0]   # short last group: amax 2 -> 2^-7
    # row 1: amax 500 -> scale 2^0 and 500 saturates to 448; 464 (a tie with 480) too
    X[1, :3] = [500.0, 464.0, -470.0]
    # row 2: all zero -> code 0, zero elements
    # row 3: a NaN poisons its group only
    X[3, :2] = [np.nan, 1.0]
    X[3, 32] = 3.0
    # row 4: an infinity
    X[4, 5] = np.inf
    Q, S = o.quantize_mxfp8(gen.f32_to_bf16_bits(X))
    assert S[0, 0] == 127 and list(Q[0, :4]) == [0x78, 0x50, 0x52, 0x58]
    assert S[0, 1] == 127 - 7 and Q[0, 32] == 0xF0 and Q[0, 39] == 0x78    # -1 and 2 at 2^-7: -128, 256
    assert S[1, 0] == 127 and list(Q[1, :3]) == [0x7E, 0x7E, 0xFE]
    assert S[2, 0] == 0 and S[2, 1] == 0 and np.all(Q[2] == 0)
    assert S[3, 0] == 255 and np.all(Q[3, :32] == 0x7F)
    assert S[3, 1] == 127 - 7 and Q[3, 32] == 0x7C                        # 3 at 2^-7: 384 = 1.5 * 2^8
    assert S[4, 0] == 255 and np.all(Q[4, :32] == 0x7F) and S[4, 1] == 0


def pin_quantize_error_bound(o):
    # dequantized elements up to 448 * scale lie within half an E4M3 step: 2^-4 relative
    # for normal results, 2^-10 * scale absolute below the smallest normal (2^-6 * scale);
    # larger ones (the scale leaves the group's amax in [256, 512) * scale) saturate to
    # exactly 448 * scale
    X = gen.matrix_bf16(64, 96, "normal", seed=351, std=0.7)
    Q, S = o.quantize_mxfp8(X)
    x = gen.bf16_bits_to_f32(X).astype(np.float64)
    d = _mx_decode(Q, S, 96)
    scale = np.repeat(np.ldexp(1.0, S.astype(np.int64) - 127), 32, axis=1)
    sat = np.abs(x) > 448.0 * scale
    assert np.any(sat)
    assert np.array_equal(d[sat], np.sign(x[sat]) * 448.0 * scale[sat])
    err_ok = np.abs(d - x) <= np.maximum(2.0 ** -4 * np.abs(x), 2.0 ** -10 * scale)
    assert np.all(err_ok[~sat])
    amax = np.abs(x).reshape(64, 3, 32).max(axis=2)
    assert np.all((np.abs(d).reshape(64, 3, 32).max(axis=2) >= 2.0 ** 8 * np.ldexp(1.0, S.astype(np.int64) - 127)))
    assert np.all(amax < 2.0 ** 9 * np.ldexp(1.0, S.astype(np.int64) - 127))


PINS = [
    pin_gemm_bruteforce_exact,
    pin_syrk_bruteforce_exact,
    pin_gemm_matches_numpy,
    pin_syrk_matches_numpy,
    pin_syr2k_bruteforce_exact,
    pin_syr2k_matches_numpy,
    pin_syr2k_invariants,
    pin_identity,
    pin_closed_forms,
    pin_transpose_identity,
    pin_syrk_is_gemm_triangle,
    pin_beta_accumulation,
    pin_alpha_scaling,
    pin_special_values,
    pin_entries_agree,
    pin_e4m3_decode_every_code,
    pin_e4m3_bruteforce_exact,
    pin_e4m3_equals_bf16_gemm_on_same_values,
    pin_e4m3_matches_numpy,
    pin_mxfp8_bruteforce_exact,
    pin_mxfp8_unit_scales_equal_e4m3,
    pin_mxfp8_matches_numpy,
    pin_mxfp8_scaling_exact,
    pin_quantize_every_code_round_trips,
    pin_quantize_matches_exact_rule,
    pin_quantize_ties_saturation_specials,
    pin_quantize_error_bound,
]
