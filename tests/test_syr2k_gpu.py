"""SYR2K parity: the CUDA path (through the C ABI) against the CPU oracle, on a GB300.

C = alpha * (op(A) op(B)^T + op(B) op(A)^T) + beta * C on one triangle. Checks
the referenced triangle against the oracle, and that the other triangle, the
padding within ldc and the rows below C are bit-identical afterwards.
"""

import itertools

import numpy as np
import pytest

import bm_inputs as gen
import oracle
from gpu_helpers import CBuffer, assert_parity, c_input_values, operand, run_syr2k, tile_samples, tile_variant, torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from blas3_tensor_core_gb300 import build
    build.build()
    assert torch().cuda.is_available()


def _mask(n, uplo):
    low = np.tril(np.ones((n, n), bool))
    return low if uplo == 0 else low.T


def _ab(n, k, trans, dist, seed, std=1.0, lo=-1.0, hi=1.0):
    rows, cols = (k, n) if trans else (n, k)
    A = operand(rows, cols, dist, seed, std, lo, hi, pad=(-cols) % 8 + 8)
    B = operand(rows, cols, dist, seed + 7, std, lo, hi, pad=(-cols) % 8 + 16)
    return A, B


# variants: automatic, single-SM 128x128 (128x256 falls back to it), SM-pair 256x256
@pytest.mark.parametrize("variant", [0, 2, 3], ids=["auto", "single128x128", "pair256x256"])
@pytest.mark.parametrize("uplo,trans", list(itertools.product((0, 1), (0, 1))))
# (320, 256): K is a whole number of two-k-block stages and n of 64-wide chunks, so both
# operands use stage-box copies on either side of the A/B swap
@pytest.mark.parametrize("n,k", [(300, 136), (256, 64), (520, 200), (320, 256)])
def test_syr2k_exact_integer(uplo, trans, n, k, variant):
    A, B = _ab(n, k, trans, "int", seed=15, lo=-8, hi=8)
    c0 = gen.integers(16, n * n, -50, 50).reshape(n, n).astype(np.float32)
    c0 = np.tril(c0) + np.tril(c0, -1).T
    ldc = n + (-n) % 4 + 4
    cbuf = CBuffer(n, n, ldc, False, init=c0)
    with tile_variant(variant):
        got, raw = run_syr2k(uplo, trans, n, k, 1.0, A, B, -1.0, cbuf)
    ref, _ = oracle.default().syr2k(uplo, trans, n, k, 1.0, A, B, -1.0, c0)
    mask = _mask(n, uplo)
    assert np.array_equal(got[mask], ref[mask])
    cbuf.assert_guard_intact(raw, mask_written=mask)


@pytest.mark.parametrize("uplo,trans", list(itertools.product((0, 1), (0, 1))))
@pytest.mark.parametrize("bf16_out", [False, True])
def test_syr2k_gaussian(uplo, trans, bf16_out):
    n, k = 400, 264
    A, B = _ab(n, k, trans, "normal", seed=27)
    c0 = gen.symmetric_f32(n, seed=28)
    c_init = gen.f32_to_bf16_bits(c0) if bf16_out else c0
    cbuf = CBuffer(n, n, n + 8, bf16_out, init=c_init)
    alpha, beta = 0.5, 1.0
    got, raw = run_syr2k(uplo, trans, n, k, alpha, A, B, beta, cbuf)
    ref, bound = oracle.default().syr2k(uplo, trans, n, k, alpha, A, B, beta, c_init)
    mask = _mask(n, uplo)
    assert_parity(got[mask], ref[mask], bound[mask], alpha, beta, c_input_values(c_init, bf16_out)[mask],
                  bf16_out, "syr2k")
    cbuf.assert_guard_intact(raw, mask_written=mask)


def test_syr2k_same_operands_is_twice_syrk():
    """SYR2K(A, A) equals 2 * SYRK(A) (both through the C ABI), exactly on integers."""
    import blas3_tensor_core_gb300 as bm
    from gpu_helpers import run_syrk
    n, k = 272, 96
    A, _ = _ab(n, k, 0, "int", seed=31, lo=-8, hi=8)
    two, raw = run_syr2k(0, 0, n, k, 1.0, A, A, 0.0, CBuffer(n, n, n, False))
    one, _ = run_syrk(0, 0, n, k, 2.0, A, 0.0, CBuffer(n, n, n, False))
    low = _mask(n, 0)
    assert np.array_equal(two[low], one[low])
    assert bm.bm_version() >= 100


def test_syr2k_alpha_zero_scales_triangle_only():
    n, k = 200, 64
    A = np.full((n, 72), gen.BF16_NAN, np.uint16)
    B = np.full((n, 72), gen.BF16_NAN, np.uint16)
    c0 = gen.symmetric_f32(n, seed=9)
    cbuf = CBuffer(n, n, 204, False, init=c0)
    got, raw = run_syr2k(1, 0, n, k, 0.0, A, B, -0.5, cbuf)
    mask = _mask(n, 1)
    assert np.array_equal(got[mask], (-0.5 * c0).astype(np.float32).astype(np.float64)[mask])
    cbuf.assert_guard_intact(raw, mask_written=mask)


def test_syr2k_large_lower_sampled():
    """C[4096, 4096] lower += A B^T + B A^T with A, B N(0, 1) [4096, 2048], fp32 C."""
    n, k = 4096, 2048
    A = operand(n, k, "normal", 1)
    B = operand(n, k, "normal", 2)
    c0 = gen.symmetric_f32(n, seed=3)
    cbuf = CBuffer(n, n, n, False, init=c0, extra_rows=1)
    got, raw = run_syr2k(0, 0, n, k, 1.0, A, B, 1.0, cbuf)
    rows, cols = tile_samples(n, n, tile_m=256, tile_n=256, per_tile=4, seed=8)
    keep = rows >= cols
    rows, cols = rows[keep], cols[keep]
    ref, bound = oracle.default().syr2k_entries(0, 0, k, 1.0, A, B, rows, cols, 1.0, c0)
    assert_parity(got[rows, cols], ref, bound, 1.0, 1.0, c0[rows, cols].astype(np.float64), False, "syr2k 4096")
    cbuf.assert_guard_intact(raw, mask_written=_mask(n, 0))


@pytest.mark.parametrize("trans", [0, 1])
def test_syr2k_split_k_exact(trans):
    """n = 512, k = 4096: every tile of the triangle is split along the 2k concatenated
    products (the split boundaries fall anywhere relative to the swap of A and B), and a
    second kernel sums them. Exact on small integers, upper triangle."""
    import blas3_tensor_core_gb300 as bm
    t = torch()
    n, k = 512, 4096
    need = bm.bm_syr2k_bf16_workspace_size(1, n, k)
    assert need > 0
    A, B = _ab(n, k, trans, "int", seed=71, lo=-4, hi=4)
    c0 = gen.integers(72, n * n, -50, 50).reshape(n, n).astype(np.float32)
    c0 = np.tril(c0) + np.tril(c0, -1).T
    ws = t.full((need // 4,), float("nan"), dtype=t.float32, device="cuda")
    cbuf = CBuffer(n, n, n + 4, False, init=c0)
    got, raw = run_syr2k(1, trans, n, k, 1.0, A, B, 1.0, cbuf, workspace=ws)
    ref, _ = oracle.default().syr2k(1, trans, n, k, 1.0, A, B, 1.0, c0)
    mask = _mask(n, 1)
    assert np.array_equal(got[mask], ref[mask])
    cbuf.assert_guard_intact(raw, mask_written=mask)
