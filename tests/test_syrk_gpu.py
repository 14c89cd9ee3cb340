"""SYRK parity: the CUDA path (through the C ABI) against the CPU oracle, on a GB300.

Checks the referenced triangle against the oracle and that the other triangle,
the padding within ldc and the rows below C are bit-identical afterwards (the
other triangle is neither read nor written).
"""

import itertools

import numpy as np
import pytest

import bm_inputs as gen
import oracle
from gpu_helpers import (VARIANT_IDS, VARIANTS, CBuffer, assert_parity, c_input_values, operand, run_syrk,
                         tile_samples, tile_variant, torch)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from blas3_tensor_core_gb300 import build
    build.build()
    assert torch().cuda.is_available()


def _mask(n, uplo):
    low = np.tril(np.ones((n, n), bool))
    return low if uplo == 0 else low.T


def _a(n, k, trans, dist, seed, std=1.0, lo=-1.0, hi=1.0):
    rows, cols = (k, n) if trans else (n, k)
    return operand(rows, cols, dist, seed, std, lo, hi, pad=(-cols) % 8 + 8)


@pytest.mark.parametrize("variant", VARIANTS, ids=VARIANT_IDS)
@pytest.mark.parametrize("uplo,trans", list(itertools.product((0, 1), (0, 1))))
@pytest.mark.parametrize("n,k", [(300, 136), (256, 64), (520, 200)])
def test_syrk_exact_integer(uplo, trans, n, k, variant):
    A = _a(n, k, trans, "int", seed=5, lo=-8, hi=8)
    c0 = gen.integers(6, n * n, -50, 50).reshape(n, n).astype(np.float32)
    c0 = np.tril(c0) + np.tril(c0, -1).T
    ldc = n + (-n) % 4 + 4
    cbuf = CBuffer(n, n, ldc, False, init=c0)
    with tile_variant(variant):
        got, raw = run_syrk(uplo, trans, n, k, 1.0, A, 1.0, cbuf)
    ref, _ = oracle.default().syrk(uplo, trans, n, k, 1.0, A, 1.0, c0)
    mask = _mask(n, uplo)
    assert np.array_equal(got[mask], ref[mask])
    cbuf.assert_guard_intact(raw, mask_written=mask)


@pytest.mark.parametrize("variant", [0, 3], ids=["auto", "pair256x256"])
@pytest.mark.parametrize("uplo,trans", list(itertools.product((0, 1), (0, 1))))
@pytest.mark.parametrize("bf16_out", [False, True])
def test_syrk_gaussian(uplo, trans, bf16_out, variant):
    n, k = 400, 264
    A = _a(n, k, trans, "normal", seed=7)
    c0 = gen.symmetric_f32(n, seed=8)
    c_init = gen.f32_to_bf16_bits(c0) if bf16_out else c0
    ldc = n + 8
    cbuf = CBuffer(n, n, ldc, bf16_out, init=c_init)
    alpha, beta = 0.5, -0.5
    with tile_variant(variant):
        got, raw = run_syrk(uplo, trans, n, k, alpha, A, beta, cbuf)
    ref, bound = oracle.default().syrk(uplo, trans, n, k, alpha, A, beta, c_init)
    mask = _mask(n, uplo)
    assert_parity(got[mask], ref[mask], bound[mask], alpha, beta, c_input_values(c_init, bf16_out)[mask],
                  bf16_out, "syrk")
    cbuf.assert_guard_intact(raw, mask_written=mask)


def test_syrk_alpha_zero_scales_triangle_only():
    n, k = 200, 64
    A = np.full((n, 72), gen.BF16_NAN, np.uint16)
    c0 = gen.symmetric_f32(n, seed=9)
    cbuf = CBuffer(n, n, 204, False, init=c0)
    got, raw = run_syrk(0, 0, n, k, 0.0, A, 3.0, cbuf)
    mask = _mask(n, 0)
    assert np.array_equal(got[mask], (3.0 * c0).astype(np.float32).astype(np.float64)[mask])
    cbuf.assert_guard_intact(raw, mask_written=mask)


def test_syrk_full_size_lower_8192x4096():
    """C[8192, 8192] = A A^T + C, A N(0, 1) [8192, 4096], C symmetric fp32 N(0, 1), lower."""
    n, k = 8192, 4096
    A = operand(n, k, "normal", 1)
    c0 = gen.symmetric_f32(n, seed=3)
    cbuf = CBuffer(n, n, n, False, init=c0, extra_rows=1)
    got, raw = run_syrk(0, 0, n, k, 1.0, A, 1.0, cbuf)
    mask = _mask(n, 0)
    rows, cols = tile_samples(n, n, per_tile=4, seed=6)
    keep = rows >= cols
    rows, cols = rows[keep], cols[keep]
    diag = np.arange(0, n, 97)
    rows = np.concatenate([rows, diag])
    cols = np.concatenate([cols, diag])
    ref, bound = oracle.default().syrk_entries(0, 0, k, 1.0, A, rows, cols, 1.0, c0)
    assert_parity(got[rows, cols], ref, bound, 1.0, 1.0, c0[rows, cols].astype(np.float64), False, "syrk 8192")
    assert np.all(np.isfinite(got[mask]))
    cbuf.assert_guard_intact(raw, mask_written=mask)
