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
                         tile_variant, torch)

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


@pytest.mark.parametrize("variant,n", [(3, 4352), (2, 2176)], ids=["pair256x256", "single128x128"])
@pytest.mark.parametrize("uplo", [0, 1], ids=["lower", "upper"])
@pytest.mark.parametrize("beta", [1.0, 0.0])
def test_syrk_grouped_order_two_groups_exact(variant, n, uplo, beta):
    """17 tile rows: the inside tiles go in a group of 16 tile rows and a group of one,
    column by column (the upper triangle in the transposed order). With beta = 1 the
    inside tiles take the group path, whose first chunk of C is loaded before the
    accumulator is ready, and the diagonal tiles the transposing path with the blocks
    outside the triangle skipped. Exact on small integers; the other triangle, the
    ldc padding and the rows below C stay bit-identical."""
    import blas3_tensor_core_gb300 as bm
    k = 136
    with tile_variant(variant):
        st, rows, cols = bm.bm_syrk_bf16_tile_order(uplo, n, k)
        assert st == 0
    tile = 256 if variant == 3 else 128
    assert (n + tile - 1) // tile == 17 and len(rows) == 17 + 17 * 16 // 2
    A = _a(n, k, 0, "int", seed=71, lo=-8, hi=8)
    c0 = gen.integers(72, n * n, -50, 50).reshape(n, n).astype(np.float32)
    c0 = np.tril(c0) + np.tril(c0, -1).T
    cbuf = CBuffer(n, n, n + 4, False, init=c0)
    with tile_variant(variant):
        got, raw = run_syrk(uplo, 0, n, k, 1.0, A, beta, cbuf)
    ref, _ = oracle.default().syrk(uplo, 0, n, k, 1.0, A, beta, c0)
    mask = _mask(n, uplo)
    assert np.array_equal(got[mask], ref[mask])
    cbuf.assert_guard_intact(raw, mask_written=mask)


@pytest.mark.parametrize("n,bf16_out,beta", [(1002, False, 1.0), (1005, True, 0.0), (2306, False, 0.0)],
                         ids=["f32_beta1", "bf16_beta0", "f32_pair"])
@pytest.mark.parametrize("uplo", [0, 1], ids=["lower", "upper"])
def test_syrk_row_end_off_16_bytes_exact(n, bf16_out, beta, uplo):
    """Rows of C that do not end on a 16-byte boundary take masked plain stores for every
    tile (a TMA store would also write the columns from n to the boundary). Exact on small
    integers; the other triangle, the columns past n and the rows below C stay unchanged."""
    k = 256
    A = _a(n, k, 0, "int", seed=73, lo=-8, hi=8)
    c0 = gen.integers(74, n * n, -50, 50).reshape(n, n).astype(np.float32)
    c0 = np.tril(c0) + np.tril(c0, -1).T
    c_init = gen.f32_to_bf16_bits(c0) if bf16_out else c0
    per = 8 if bf16_out else 4
    cbuf = CBuffer(n, n, n + (-n) % per + per, bf16_out, init=c_init)
    got, raw = run_syrk(uplo, 0, n, k, 1.0, A, beta, cbuf)
    ref, _ = oracle.default().syrk(uplo, 0, n, k, 1.0, A, beta, c_init if beta != 0.0 else None)
    if bf16_out:
        ref = gen.bf16_bits_to_f32(gen.f32_to_bf16_bits(ref.astype(np.float32))).astype(np.float64)
    mask = _mask(n, uplo)
    assert np.array_equal(got[mask], ref[mask])
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


def _random_workspace(nbytes, seed):
    t = torch()
    ws = t.empty((nbytes // 4,), dtype=t.float32, device="cuda")
    g = t.Generator(device="cuda")
    g.manual_seed(seed)
    ws.view(t.int32).copy_(t.randint(-2**31, 2**31 - 1, (nbytes // 4,), dtype=t.int32, device="cuda", generator=g))
    return ws


@pytest.mark.parametrize("uplo,trans", list(itertools.product((0, 1), (0, 1))))
def test_syrk_split_k_small_n_long_k_exact(uplo, trans):
    """n = 512, k = 8192: the 6 tiles of the triangle cannot fill the GPU, so every tile is
    split along K into the workspace (filled with random bits first) and a second kernel
    sums the partials, writing only the triangle. Exact on small integers, twice in a row."""
    import blas3_tensor_core_gb300 as bm
    n, k = 512, 8192
    need = bm.bm_syrk_bf16_workspace_size(uplo, n, k)
    plan = bm.bm_syrk_bf16_plan(uplo, n, k, need)[1]
    assert plan.k_splits > 1 and plan.kernels == 2
    A = _a(n, k, trans, "int", seed=41, lo=-4, hi=4)
    c0 = gen.integers(42, n * n, -50, 50).reshape(n, n).astype(np.float32)
    c0 = np.tril(c0) + np.tril(c0, -1).T
    ws = _random_workspace(need, 43)
    ref, _ = oracle.default().syrk(uplo, trans, n, k, 1.0, A, -1.0, c0)
    mask = _mask(n, uplo)
    for _ in range(2):
        cbuf = CBuffer(n, n, n + 4, False, init=c0)
        got, raw = run_syrk(uplo, trans, n, k, 1.0, A, -1.0, cbuf, workspace=ws)
        assert np.array_equal(got[mask], ref[mask])
        cbuf.assert_guard_intact(raw, mask_written=mask)


@pytest.mark.parametrize("uplo", [0, 1], ids=["lower", "upper"])
def test_syrk_tail_split_summed_in_kernel_exact(uplo):
    """n = 3072 on SM pairs: 12 * 13 / 2 = 78 tiles = 76 + 2; the 2 tiles of the last wave
    are split along K and summed inside the kernel (with beta folded into split 0), which
    writes only the triangle. Exact on small integers, with a workspace of random bits."""
    import blas3_tensor_core_gb300 as bm
    n, k = 3072, 4096
    need = bm.bm_syrk_bf16_workspace_size(uplo, n, k)
    plan = bm.bm_syrk_bf16_plan(uplo, n, k, need)[1]
    assert plan.cta_pair == 2 and plan.tiles == 78
    assert plan.split_tiles == 2 and plan.k_splits > 1 and plan.kernels == 1
    A = _a(n, k, 0, "int", seed=51, lo=-3, hi=3)
    c0 = gen.integers(52, n * n, -50, 50).reshape(n, n).astype(np.float32)
    c0 = np.tril(c0) + np.tril(c0, -1).T
    ws = _random_workspace(need, 53)
    cbuf = CBuffer(n, n, n, False, init=c0)
    got, raw = run_syrk(uplo, 0, n, k, 1.0, A, 1.0, cbuf, workspace=ws)
    ref, _ = oracle.default().syrk(uplo, 0, n, k, 1.0, A, 1.0, c0)
    mask = _mask(n, uplo)
    assert np.array_equal(got[mask], ref[mask])
    cbuf.assert_guard_intact(raw, mask_written=mask)


@pytest.mark.parametrize("bf16_out", [False, True])
def test_syrk_split_k_gaussian_beta(bf16_out):
    import blas3_tensor_core_gb300 as bm
    n, k = 400, 8000
    need = bm.bm_syrk_bf16_workspace_size(0, n, k)
    assert bm.bm_syrk_bf16_plan(0, n, k, need)[1].k_splits > 1
    A = _a(n, k, 1, "normal", seed=61)
    c0 = gen.symmetric_f32(n, seed=62)
    c_init = gen.f32_to_bf16_bits(c0) if bf16_out else c0
    cbuf = CBuffer(n, n, n + 8, bf16_out, init=c_init)
    got, raw = run_syrk(0, 1, n, k, 0.5, A, -1.5, cbuf, workspace=_random_workspace(need, 63))
    ref, bound = oracle.default().syrk(0, 1, n, k, 0.5, A, -1.5, c_init)
    mask = _mask(n, 0)
    assert_parity(got[mask], ref[mask], bound[mask], 0.5, -1.5, c_input_values(c_init, bf16_out)[mask], bf16_out,
                  "syrk split")
    cbuf.assert_guard_intact(raw, mask_written=mask)
