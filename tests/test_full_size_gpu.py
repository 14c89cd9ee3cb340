"""Whole-output parity at full size: every configured workload, every element of C,
through the C ABI in the launch plan the bench times (with the workspace the
planner asks for), against the CPU oracle, on a GB300.

Workloads (synthetic, seeded; see the input recipe): the 256^3 uniform GEMM into
FP32 C, the 4096^3 GEMM into bf16 C, the K-sweep (K in 256 .. 8192 crossed with
M = N in {512, 4096}), the backward pair (dX = dY W; dW += dY^T X with beta = 1
into a bf16 C), lower SYRK 8192 x 4096 with beta = 1 into a symmetric FP32 C
(plus the untouched upper triangle and guard band, bitwise), lower SYR2K of the
same size, and the FP8 E4M3 and MXFP8 GEMMs at 4096^3. Each test prints the
worst |err| / tolerance it saw (run with -s to see them).
"""

import numpy as np
import pytest

import bm_inputs as gen
import oracle
from gpu_helpers import (CBuffer, assert_parity, c_input_values, operand, run_gemm, run_gemm_e4m3, run_gemm_mxfp8,
                         run_syr2k, run_syrk, torch)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from blas3_tensor_core_gb300 import build
    build.build()
    assert torch().cuda.is_available()


def _workspace(nbytes):
    t = torch()
    return t.empty((max(nbytes // 4, 1),), dtype=t.float32, device="cuda") if nbytes else None


def _stored(rows, cols, trans):
    return (cols, rows) if trans else (rows, cols)


GEMMS = [
    # name, m, n, k, transA, transB, distribution, std, beta, bf16 C
    ("gemm_256x256x256_uniform_f32c", 256, 256, 256, 0, 0, "uniform", 1.0, 0.0, False),
    ("gemm_bf16_4096x4096x4096_nn_bf16c", 4096, 4096, 4096, 0, 0, "normal", 1.0, 0.0, True),
    ("sweep_512x512x256", 512, 512, 256, 0, 0, "normal", 1.0, 0.0, True),
    ("sweep_512x512x512", 512, 512, 512, 0, 0, "normal", 1.0, 0.0, True),
    ("sweep_512x512x1024", 512, 512, 1024, 0, 0, "normal", 1.0, 0.0, True),
    ("sweep_512x512x4096", 512, 512, 4096, 0, 0, "normal", 1.0, 0.0, True),
    ("sweep_512x512x8192", 512, 512, 8192, 0, 0, "normal", 1.0, 0.0, True),
    ("sweep_4096x4096x256", 4096, 4096, 256, 0, 0, "normal", 1.0, 0.0, True),
    ("sweep_4096x4096x512", 4096, 4096, 512, 0, 0, "normal", 1.0, 0.0, True),
    ("sweep_4096x4096x1024", 4096, 4096, 1024, 0, 0, "normal", 1.0, 0.0, True),
    ("sweep_4096x4096x8192", 4096, 4096, 8192, 0, 0, "normal", 1.0, 0.0, True),
    ("bwd_dX_2048x5120x5120", 2048, 5120, 5120, 0, 0, "normal", 0.02, 0.0, True),
    ("bwd_dW_5120x5120x2048_transA_beta1", 5120, 5120, 2048, 1, 0, "normal", 0.02, 1.0, True),
]


@pytest.mark.parametrize("name,m,n,k,ta,tb,dist,std,beta,cbf", GEMMS, ids=[g[0] for g in GEMMS])
def test_gemm_whole_output(name, m, n, k, ta, tb, dist, std, beta, cbf):
    import blas3_tensor_core_gb300 as bm
    A = operand(*_stored(m, k, ta), dist, 1, std)
    B = operand(*_stored(k, n, tb), dist, 2, std)
    c_init = gen.matrix_bf16(m, n, "normal", 3, std) if beta != 0 else None
    cbuf = CBuffer(m, n, n, cbf, init=c_init, extra_rows=1)
    ws = _workspace(bm.bm_gemm_bf16_workspace_size(m, n, k))
    got, raw = run_gemm(m, n, k, ta, tb, 1.0, A, B, beta, cbuf, workspace=ws)
    ref, bound = oracle.default().gemm(m, n, k, ta, tb, 1.0, A, B, beta, c_init)
    worst = assert_parity(got, ref, bound, 1.0, beta, c_input_values(c_init, cbf), cbf, name)
    print(f"{name}: whole output, worst |err|/tol = {worst:.4g}")
    cbuf.assert_guard_intact(raw)


def _lower(n):
    return np.tril(np.ones((n, n), bool))


def test_syrk_lower_8192x4096_whole_triangle():
    """C[8192, 8192] = A A^T + C, A N(0, 1) [8192, 4096], C symmetric FP32 N(0, 1), lower."""
    import blas3_tensor_core_gb300 as bm
    n, k = 8192, 4096
    A = operand(n, k, "normal", 1)
    c0 = gen.symmetric_f32(n, seed=3)
    cbuf = CBuffer(n, n, n, False, init=c0, extra_rows=1)
    ws = _workspace(bm.bm_syrk_bf16_workspace_size(bm.BM_LOWER, n, k))
    got, raw = run_syrk(0, 0, n, k, 1.0, A, 1.0, cbuf, workspace=ws)
    ref, bound = oracle.default().syrk(0, 0, n, k, 1.0, A, 1.0, c0)
    mask = _lower(n)
    worst = assert_parity(got[mask], ref[mask], bound[mask], 1.0, 1.0, c0.astype(np.float64)[mask], False,
                          "syrk 8192x4096")
    print(f"syrk_lower_8192x4096_f32c_beta1: whole triangle, worst |err|/tol = {worst:.4g}")
    cbuf.assert_guard_intact(raw, mask_written=mask)


def test_syr2k_lower_8192x4096_whole_triangle():
    import blas3_tensor_core_gb300 as bm
    n, k = 8192, 4096
    A = operand(n, k, "normal", 1)
    B = operand(n, k, "normal", 2)
    c0 = gen.symmetric_f32(n, seed=3)
    cbuf = CBuffer(n, n, n, False, init=c0, extra_rows=1)
    ws = _workspace(bm.bm_syr2k_bf16_workspace_size(bm.BM_LOWER, n, k))
    got, raw = run_syr2k(0, 0, n, k, 1.0, A, B, 1.0, cbuf, workspace=ws)
    ref, bound = oracle.default().syr2k(0, 0, n, k, 1.0, A, B, 1.0, c0)
    mask = _lower(n)
    worst = assert_parity(got[mask], ref[mask], bound[mask], 1.0, 1.0, c0.astype(np.float64)[mask], False,
                          "syr2k 8192x4096")
    print(f"syr2k_lower_8192x4096_f32c_beta1: whole triangle, worst |err|/tol = {worst:.4g}")
    cbuf.assert_guard_intact(raw, mask_written=mask)


def test_e4m3_4096_whole_output():
    import blas3_tensor_core_gb300 as bm
    m = n = k = 4096
    A = gen.matrix_e4m3(m, k, "normal", seed=1)
    B = gen.matrix_e4m3(n, k, "normal", seed=2)
    cbuf = CBuffer(m, n, n, True, extra_rows=1)
    ws = _workspace(bm.bm_gemm_e4m3_workspace_size(m, n, k))
    got, raw = run_gemm_e4m3(m, n, k, 1.0, A, B, 0.0, cbuf, workspace=ws)
    ref, bound = oracle.default().gemm_e4m3(m, n, k, 1.0, A, B)
    worst = assert_parity(got, ref, bound, 1.0, 0.0, None, True, "e4m3 4096^3")
    print(f"gemm_e4m3_4096x4096x4096_tn_bf16c: whole output, worst |err|/tol = {worst:.4g}")
    cbuf.assert_guard_intact(raw)


def test_mxfp8_4096_whole_output():
    """MXFP8 operands as produced by quantizing N(0, 1) data: E4M3 codes of N(0, 1) values and
    UE8M0 group scales of 2^-3 .. 2^3."""
    import blas3_tensor_core_gb300 as bm
    m = n = k = 4096
    A = gen.matrix_e4m3(m, k, "normal", seed=1)
    B = gen.matrix_e4m3(n, k, "normal", seed=2)
    SA = gen.integers(3, m * (k // 32), 124, 130).reshape(m, k // 32).astype(np.uint8)
    SB = gen.integers(4, n * (k // 32), 124, 130).reshape(n, k // 32).astype(np.uint8)
    cbuf = CBuffer(m, n, n, True, extra_rows=1)
    ws = _workspace(bm.bm_gemm_mxfp8_workspace_size(m, n, k))
    got, raw = run_gemm_mxfp8(m, n, k, 1.0, A, SA, B, SB, 0.0, cbuf, workspace=ws)
    ref, bound = oracle.default().gemm_mxfp8(m, n, k, 1.0, A, SA, B, SB)
    worst = assert_parity(got, ref, bound, 1.0, 0.0, None, True, "mxfp8 4096^3")
    print(f"gemm_mxfp8_4096x4096x4096_tn_bf16c: whole output, worst |err|/tol = {worst:.4g}")
    cbuf.assert_guard_intact(raw)
