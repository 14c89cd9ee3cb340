"""FP8 E4M3 GEMM parity (C = alpha * A B^T + beta * C): the CUDA path through the
C ABI against the CPU oracle, on a GB300.

Exact-integer inputs (|x| <= 8, exact in E4M3) pin the kind::f8f6f4 instruction
descriptor and the 128-element k-blocks bit for bit on every tile variant;
Gaussian inputs use the tolerance 1e-3 * |alpha| * sum|a*b| (+ 2^-8 |ref| for
BF16 output).
"""

import numpy as np
import pytest

import bm_inputs as gen
import oracle
from gpu_helpers import (VARIANT_IDS, VARIANTS, CBuffer, assert_parity, c_input_values, run_gemm_e4m3, tile_samples,
                         tile_variant, torch)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from blas3_tensor_core_gb300 import build
    build.build()
    assert torch().cuda.is_available()


def _codes(rows, cols, dist, seed, std=1.0, lo=-8, hi=8):
    codes = gen.matrix_e4m3(rows, cols, dist, seed, std, lo, hi)
    pad = (-cols) % 16 + 16
    return gen.pad_ld(codes, cols + pad, np.uint8(0x7F))  # NaN padding: never read


def _ldc(n, bf16):
    per = 8 if bf16 else 4
    return n + (-n) % per + per


@pytest.mark.parametrize("variant", VARIANTS, ids=VARIANT_IDS)
@pytest.mark.parametrize("shape", [(256, 256, 256), (200, 300, 136), (129, 520, 64), (1, 8, 16), (520, 264, 200)])
def test_e4m3_exact_integer_bitwise(shape, variant):
    m, n, k = shape
    A = _codes(m, k, "int", 5)
    B = _codes(n, k, "int", 6)
    cbuf = CBuffer(m, n, _ldc(n, False), False, init=np.full((m, n), np.nan, np.float32))
    with tile_variant(variant):
        got, raw = run_gemm_e4m3(m, n, k, 1.0, A, B, 0.0, cbuf)
    ref, _ = oracle.default().gemm_e4m3(m, n, k, 1.0, A, B)
    assert np.array_equal(got, ref), f"max |diff| {np.max(np.abs(got - ref))}"
    cbuf.assert_guard_intact(raw)


@pytest.mark.parametrize("bf16_out,beta", [(False, 0.0), (False, 1.0), (True, 0.0), (True, -0.5)])
def test_e4m3_gaussian_ragged(bf16_out, beta):
    m, n, k = 640, 520, 392
    A = _codes(m, k, "normal", 11)
    B = _codes(n, k, "normal", 12, std=0.25)
    c0 = gen.matrix_f32(m, n, "normal", seed=13)
    c_init = gen.f32_to_bf16_bits(c0) if bf16_out else c0
    cbuf = CBuffer(m, n, _ldc(n, bf16_out), bf16_out, init=c_init)
    got, raw = run_gemm_e4m3(m, n, k, 0.75, A, B, beta, cbuf)
    ref, bound = oracle.default().gemm_e4m3(m, n, k, 0.75, A, B, beta, c_init if beta != 0 else None)
    assert_parity(got, ref, bound, 0.75, beta, c_input_values(c_init, bf16_out), bf16_out, "e4m3 ragged")
    cbuf.assert_guard_intact(raw)


def test_e4m3_split_k_and_deterministic():
    import blas3_tensor_core_gb300 as bm
    t = torch()
    m, n, k = 512, 512, 16384
    A = _codes(m, k, "normal", 21)
    B = _codes(n, k, "normal", 22)
    need = bm.bm_gemm_e4m3_workspace_size(m, n, k)
    assert need > 0
    ws = t.empty(need // 4, dtype=t.float32, device="cuda")
    outs = []
    for _ in range(2):
        cbuf = CBuffer(m, n, n, True)
        got, raw = run_gemm_e4m3(m, n, k, 1.0, A, B, 0.0, cbuf, workspace=ws)
        cbuf.assert_guard_intact(raw)
        outs.append(got)
    assert np.array_equal(outs[0], outs[1])
    rows, cols = tile_samples(m, n, per_tile=64, seed=7)
    ref, bound = oracle.default().gemm_e4m3_entries(k, 1.0, A, B, rows, cols)
    assert_parity(outs[0][rows, cols], ref, bound, 1.0, 0.0, None, True, "e4m3 split-K")


def test_e4m3_tail_split_summed_in_kernel():
    """80 pair tiles = 76 + 4: the 4 tail tiles split 13 ways along K (the 16 MiB tail budget) and summed inside the kernel."""
    import blas3_tensor_core_gb300 as bm
    t = torch()
    m, n, k = 2560, 2048, 8192
    A = _codes(m, k, "normal", 23)
    B = _codes(n, k, "normal", 24)
    need = bm.bm_gemm_e4m3_workspace_size(m, n, k)
    ws = t.empty(need // 4, dtype=t.float32, device="cuda")
    cbuf = CBuffer(m, n, n, True)
    got, raw = run_gemm_e4m3(m, n, k, 1.0, A, B, 0.0, cbuf, workspace=ws)
    cbuf.assert_guard_intact(raw)
    # the split tiles are in the last tile column; columns 1823, 1919, 1951 and 2047 fall in
    # tile-local 32-column chunks 0, 3, 4 and 7, so both epilogue halves of every row are checked
    band_c = np.repeat(np.array([n - 225, n - 129, n - 97, n - 1]), m)
    band_r = np.tile(np.arange(m), 4)
    rows, cols = tile_samples(m, n, per_tile=16, seed=8, extra=(band_r, band_c))
    ref, bound = oracle.default().gemm_e4m3_entries(k, 1.0, A, B, rows, cols)
    assert_parity(got[rows, cols], ref, bound, 1.0, 0.0, None, True, "e4m3 tail split")


@pytest.mark.parametrize("bf16_out,beta", [(False, 0.0), (True, -1.0)])
def test_e4m3_n_half_tail_whole_output_exact(bf16_out, beta):
    """80 pair tiles = 76 + 4 with too few k-blocks for a K split: the 4 tail tiles run as
    two units of half their columns each (MMA N = 128 over half of each CTA's B rows), no
    partial sums. Small integers (exact in E4M3) make every element exact, so the whole
    output is compared with the oracle."""
    m, n, k = 2560, 2048, 1024
    A = _codes(m, k, "int", 31, lo=-4, hi=4)
    B = _codes(n, k, "int", 32, lo=-4, hi=4)
    c0 = gen.integers(33, m * n, -30, 30).reshape(m, n).astype(np.float32)
    c_init = gen.f32_to_bf16_bits(c0) if bf16_out else c0
    cbuf = CBuffer(m, n, _ldc(n, bf16_out), bf16_out, init=c_init)
    got, raw = run_gemm_e4m3(m, n, k, 1.0, A, B, beta, cbuf)
    cbuf.assert_guard_intact(raw)
    ref, _ = oracle.default().gemm_e4m3(m, n, k, 1.0, A, B, beta, c_init if beta != 0.0 else None)
    if bf16_out:
        ref = gen.bf16_bits_to_f32(gen.f32_to_bf16_bits(ref.astype(np.float32))).astype(np.float64)
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("m,n,k,bf16_out,beta", [(520, 262, 200, False, 0.0), (2304, 2309, 256, True, -1.0)],
                         ids=["single_f32", "pair_bf16_beta"])
def test_e4m3_row_end_off_16_bytes_exact(m, n, k, bf16_out, beta):
    """Rows of C that do not end on a 16-byte boundary are stored with masked plain stores
    (a TMA store would also write the columns from n to the boundary). Exact integers: the
    whole output equals the oracle, and the columns past n and the rows below C are unchanged."""
    A = _codes(m, k, "int", 21)
    B = _codes(n, k, "int", 22)
    c0 = gen.integers(23, m * n, -30, 30).reshape(m, n).astype(np.float32)
    c_init = gen.f32_to_bf16_bits(c0) if bf16_out else c0
    cbuf = CBuffer(m, n, _ldc(n, bf16_out), bf16_out, init=c_init)
    got, raw = run_gemm_e4m3(m, n, k, 1.0, A, B, beta, cbuf)
    cbuf.assert_guard_intact(raw)
    ref, _ = oracle.default().gemm_e4m3(m, n, k, 1.0, A, B, beta, c_init if beta != 0 else None)
    if bf16_out:
        ref = gen.bf16_bits_to_f32(gen.f32_to_bf16_bits(ref.astype(np.float32))).astype(np.float64)
    assert np.array_equal(got, ref)
