"""Plant plausible mistakes in copies of the oracle's C source; each must fail a pin.

This shows the pins are strong enough to catch a dropped term, a wrong sign, a
transposed operand or index, a wrong triangle or a broken BLAS convention
anywhere in the oracle. The mutants are compiled into a temporary directory;
the committed oracle is never modified.
"""

import os

import pytest

import oracle
from oracle_pins import PINS

SRC = os.path.join(os.path.dirname(oracle.__file__), "bm_oracle.c")

# (name, text to replace, replacement, which occurrence: 0 = first)
MUTANTS = [
    ("gemm_sign", "acc += prod;", "acc -= prod;", 0),
    ("syrk_sign", "acc += prod;", "acc -= prod;", 1),
    ("gemm_drop_alpha", "double value = alpha * acc;", "double value = acc;", 0),
    ("syrk_drop_alpha", "double value = alpha * acc;", "double value = acc;", 1),
    ("gemm_drop_beta", "value += beta * c_input", "value += c_input", 0),
    ("syrk_drop_beta_term", "value += beta * c_input", "value += 0.0 * c_input", 1),
    ("ignore_transpose", "return bf16_value(X[c * ld + r]);", "return bf16_value(X[r * ld + c]);", 0),
    ("transposed_c_input", "((const float *)C)[i * ldc + j]", "((const float *)C)[j * ldc + i]", 0),
    ("gemm_drop_first_term", "for (int64_t p = 0; p < k; ++p) {", "for (int64_t p = 1; p < k; ++p) {", 0),
    ("syrk_drop_last_term", "for (int64_t p = 0; p < k; ++p) {", "for (int64_t p = 0; p + 1 < k; ++p) {", 1),
    ("gemm_signed_bound", "mag += fabs(prod);", "mag += prod;", 0),
    ("lower_strict", "return uplo == 0 ? (i >= j) : (i <= j);", "return uplo == 0 ? (i > j) : (i <= j);", 0),
    ("upper_as_lower", "return uplo == 0 ? (i >= j) : (i <= j);", "return (i >= j);", 0),
    ("syrk_same_row_twice", "op_at(A, lda, trans, j, p)", "op_at(A, lda, trans, i, p)", 0),
    ("negative_beta_dropped", "if (beta != 0.0)\n        value += beta", "if (beta > 0.0)\n        value += beta", 0),
    ("alpha_zero_reads_a", "if (alpha != 0.0) {\n        for", "{\n        for", 0),
    ("bf16_c_misread", "return bf16_value(((const uint16_t *)C)[i * ldc + j]);",
     "return (double)((const float *)C)[i * ldc + j];", 0),
    ("syr2k_drop_second_product", "ba += y;", "ba += 0.0 * y;", 0),
    ("syr2k_same_operand_twice", "op_at(A, lda, trans, i, p) * op_at(B, ldb, trans, j, p)",
     "op_at(A, lda, trans, i, p) * op_at(A, lda, trans, j, p)", 0),
    ("syr2k_mirrored_second_product", "op_at(B, ldb, trans, i, p) * op_at(A, lda, trans, j, p)",
     "op_at(A, lda, trans, i, p) * op_at(B, ldb, trans, j, p)", 0),
    ("syr2k_drop_beta", "value += beta * c_input", "value += 0.0 * c_input", 2),
    ("syr2k_signed_bound", "mag += fabs(x) + fabs(y);", "mag += fabs(x) + y;", 0),
    ("e4m3_bias_off_by_one", "mag = ldexp(1.0 + (double)m / 8.0, e - 7);", "mag = ldexp(1.0 + (double)m / 8.0, e - 8);", 0),
    ("e4m3_no_subnormals", "mag = ldexp((double)m / 8.0, -6);", "mag = ldexp(1.0 + (double)m / 8.0, -7);", 0),
    ("e4m3_mantissa_bits", "int e = (code >> 3) & 0xF, m = code & 7;", "int e = (code >> 3) & 0xF, m = code & 3;", 0),
    ("e4m3_sign_dropped", "return (code & 0x80) ? -mag : mag;", "return mag;", 0),
    ("e4m3_b_k_reversed", "e4m3_value(B[j * ldb + p])", "e4m3_value(B[j * ldb + (k - 1 - p)])", 0),
    ("gemm_last_column_skipped", "for (int64_t j = 0; j < n; ++j)\n            gemm_element",
     "for (int64_t j = 0; j + 1 < n; ++j)\n            gemm_element", 0),
    # MXFP8 GEMM
    ("mx_group_of_16", "SA[i * ldsa + p / 32]", "SA[i * ldsa + p / 16]", 0),
    ("mx_b_scale_of_row_i", "SB[j * ldsb + p / 32]", "SB[i * ldsb + p / 32]", 0),
    ("mx_b_scale_dropped", " * ue8m0_value(SB[j * ldsb + p / 32])", "", 0),
    ("mx_scale_bias_128", "return ldexp(1.0, (int)code - 127);", "return ldexp(1.0, (int)code - 128);", 0),
    ("mx_scale_ld_ignored", "SA[i * ldsa + p / 32]", "SA[i * ((k + 31) / 32) + p / 32]", 0),
    ("mx_group_index_mod", "SB[j * ldsb + p / 32]", "SB[j * ldsb + p % 32 / 8]", 0),
    ("mx_signed_bound", "            acc += prod;\n            mag += fabs(prod);\n        }\n    }\n    double value = alpha * acc;\n    if (beta != 0.0)\n        value += beta * c_input(C, ldc, c_is_bf16, i, j);\n    *ref = value;\n    *bound = mag;\n}\n\n/* One output element of SYR2K",
     "            acc += prod;\n            mag += prod;\n        }\n    }\n    double value = alpha * acc;\n    if (beta != 0.0)\n        value += beta * c_input(C, ldc, c_is_bf16, i, j);\n    *ref = value;\n    *bound = mag;\n}\n\n/* One output element of SYR2K", 0),
    # MXFP8 quantization (OCP MX conversion)
    ("q_emax_7", "e = (ex - 1) - 8;", "e = (ex - 1) - 7;", 0),
    ("q_ceil_log2", "e = (ex - 1) - 8;", "e = ex - 8;", 0),
    ("q_ties_away", "(err == best_err && (c & 1) == 0)", "(err == best_err)", 0),
    ("q_ties_down", "(err == best_err && (c & 1) == 0)", "(0)", 0),
    ("q_no_saturation", "        best = 0x7E;\n", "        best = 0x7F;\n", 0),
    ("q_sign_dropped", "return (uint8_t)(signbit(y) ? (best | 0x80) : best);", "return (uint8_t)best;", 0),
    ("q_signed_amax", "else if (fabs(x) > amax)\n                    amax = fabs(x);", "else if (x > amax)\n                    amax = x;", 0),
    ("q_zero_group_code", "int e = -127;\n            if (amax > 0.0) {", "int e = 0;\n            if (amax > 0.0) {", 0),
    ("q_specials_ignored", "special = 1;", "special = 0;", 0),
    ("q_no_low_clamp", "if (e < -127)\n                    e = -127;", "if (e < -200)\n                    e = -127;", 0),
    ("q_amax_half_group", "for (int64_t p = p0; p < p1; ++p) {\n                double x = bf16_value",
     "for (int64_t p = p0; p < p1 && p < p0 + 16; ++p) {\n                double x = bf16_value", 0),
]


def _mutate(text, old, new, occurrence):
    start = -1
    for _ in range(occurrence + 1):
        start = text.find(old, start + 1)
        assert start >= 0, f"mutation anchor not found: {old!r}"
    return text[:start] + new + text[start + len(old):]


@pytest.mark.parametrize("name,old,new,occ", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, name, old, new, occ):
    src = open(SRC).read()
    mutated = _mutate(src, old, new, occ)
    assert mutated != src
    path = tmp_path / f"{name}.c"
    path.write_text(mutated)
    lib = oracle.compile_oracle(str(path), str(tmp_path / f"lib{name}.so"))
    o = oracle.Oracle(lib)
    failures = []
    for pin in PINS:
        try:
            pin(o)
        except Exception:  # any failure of a pin counts as catching the mutant
            failures.append(pin.__name__)
    assert failures, f"mutant {name} passed every pin"
