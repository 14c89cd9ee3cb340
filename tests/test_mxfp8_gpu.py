"""MXFP8 block-scaled GEMM parity (C = alpha * (A . SA)(B . SB)^T + beta * C): the CUDA
path through the C ABI against the CPU oracle, on a GB300.

A and B hold E4M3 codes; every group of 32 consecutive elements of a row along K
has its own UE8M0 scale. Exact-integer data (|x| <= 8) with scales 2^-1, 2^0 and
2^1 keep every FP32 partial sum exact, so the scale-factor layout in shared and
tensor memory and the per-MMA choice of scale byte are pinned bit for bit on
every tile variant; Gaussian data with scales 2^-7 .. 2^7 use the tolerance
1e-3 * |alpha| * sum|a*b| (+ 2^-8 |ref| for BF16 output).
"""

import numpy as np
import pytest

import bm_inputs as gen
import oracle
from gpu_helpers import (CBuffer, assert_parity, c_input_values, run_gemm_mxfp8, tile_samples, tile_variant,
                         torch)

pytestmark = pytest.mark.gpu

# automatic choice, 128 x 128 tiles on single SMs, 256 x 128 tiles on SM pairs
MX_VARIANTS = [0, 1, 3]
MX_IDS = ["auto", "single128x128", "pair256x128"]


@pytest.fixture(scope="module", autouse=True)
def _built():
    from blas3_tensor_core_gb300 import build
    build.build()
    assert torch().cuda.is_available()


def _codes(rows, cols, dist, seed, std=1.0, lo=-8, hi=8):
    codes = gen.matrix_e4m3(rows, cols, dist, seed, std, lo, hi)
    pad = (-cols) % 16 + 16
    return gen.pad_ld(codes, cols + pad, np.uint8(0x7F))  # NaN padding: never read


def _scales(rows, k, seed, lo, hi):
    groups = (k + 31) // 32
    return gen.integers(seed, rows * groups, lo, hi).reshape(rows, groups).astype(np.uint8)


def _ldc(n, bf16):
    per = 8 if bf16 else 4
    return n + (-n) % per + per


def _explain(got, ref):
    bad = np.argwhere(got != ref)
    i, j = bad[0]
    return f"{len(bad)} of {got.size} differ; first at {(int(i), int(j))}: got {got[i, j]!r} ref {ref[i, j]!r}"


@pytest.mark.parametrize("variant", MX_VARIANTS, ids=MX_IDS)
@pytest.mark.parametrize("shape", [(256, 256, 256), (200, 300, 136), (129, 520, 64), (1, 16, 32), (520, 264, 200),
                                   (384, 256, 1024)])
def test_mxfp8_exact_integer_bitwise(shape, variant):
    m, n, k = shape
    A = _codes(m, k, "int", 5)
    B = _codes(n, k, "int", 6)
    SA = _scales(m, k, 7, 126, 128)
    SB = _scales(n, k, 8, 126, 128)
    cbuf = CBuffer(m, n, _ldc(n, False), False, init=np.full((m, n), np.nan, np.float32))
    with tile_variant(variant):
        got, raw = run_gemm_mxfp8(m, n, k, 1.0, A, SA, B, SB, 0.0, cbuf, pad_code=0x7F)
    ref, _ = oracle.default().gemm_mxfp8(m, n, k, 1.0, A, SA, B, SB)
    assert np.array_equal(got, ref), _explain(got, ref)
    cbuf.assert_guard_intact(raw)


@pytest.mark.parametrize("variant", [0, 3], ids=["auto", "pair256x128"])
@pytest.mark.parametrize("bf16_out,beta", [(False, 0.0), (False, 1.0), (True, 0.0), (True, -0.5)])
def test_mxfp8_gaussian_ragged(bf16_out, beta, variant):
    m, n, k = 640, 520, 392
    A = _codes(m, k, "normal", 11)
    B = _codes(n, k, "normal", 12, std=0.25)
    SA = _scales(m, k, 13, 120, 134)
    SB = _scales(n, k, 14, 120, 134)
    c0 = gen.matrix_f32(m, n, "normal", seed=15)
    c_init = gen.f32_to_bf16_bits(c0) if bf16_out else c0
    cbuf = CBuffer(m, n, _ldc(n, bf16_out), bf16_out, init=c_init)
    with tile_variant(variant):
        got, raw = run_gemm_mxfp8(m, n, k, 0.75, A, SA, B, SB, beta, cbuf)
    ref, bound = oracle.default().gemm_mxfp8(m, n, k, 0.75, A, SA, B, SB, beta, c_init if beta != 0 else None)
    assert_parity(got, ref, bound, 0.75, beta, c_input_values(c_init, bf16_out), bf16_out, "mxfp8 ragged")
    cbuf.assert_guard_intact(raw)


def test_mxfp8_split_k_exact_and_deterministic():
    """512 x 520 output, K = 8192: too few tiles for the GPU, so every tile is split along K."""
    import blas3_tensor_core_gb300 as bm
    t = torch()
    m, n, k = 512, 520, 8192
    need = bm.bm_gemm_mxfp8_workspace_size(m, n, k)
    st, plan = bm.bm_gemm_mxfp8_plan(m, n, k, need)
    assert st == 0 and plan.k_splits > 1 and plan.tile_k == 128
    A = _codes(m, k, "int", 21, lo=-4, hi=4)
    B = _codes(n, k, "int", 22, lo=-4, hi=4)
    SA = _scales(m, k, 23, 126, 128)
    SB = _scales(n, k, 24, 126, 128)
    ws = t.full((need // 4 + 64,), float("nan"), dtype=t.float32, device="cuda")
    outs = []
    for _ in range(2):
        cbuf = CBuffer(m, n, _ldc(n, False), False, init=np.full((m, n), np.nan, np.float32))
        got, raw = run_gemm_mxfp8(m, n, k, 1.0, A, SA, B, SB, 0.0, cbuf, workspace=ws)
        cbuf.assert_guard_intact(raw)
        outs.append(got)
    assert np.array_equal(outs[0], outs[1])
    ref, _ = oracle.default().gemm_mxfp8(m, n, k, 1.0, A, SA, B, SB)
    assert np.array_equal(outs[0], ref), _explain(outs[0], ref)


def test_mxfp8_tail_split_beta_bf16():
    """4096 x 4096 x 2048 on SM pairs: 512 tiles of 256 x 128 = 6 waves of 76 + 56; whole-output
    parity with beta into a bf16 C."""
    import blas3_tensor_core_gb300 as bm
    t = torch()
    m = n = 4096
    k = 2048
    A = _codes(m, k, "normal", 31)
    B = _codes(n, k, "normal", 32)
    SA = _scales(m, k, 33, 122, 132)
    SB = _scales(n, k, 34, 122, 132)
    c_init = gen.matrix_bf16(m, n, "normal", seed=35)
    need = bm.bm_gemm_mxfp8_workspace_size(m, n, k)
    ws = t.empty((max(need // 4, 1),), dtype=t.float32, device="cuda")
    cbuf = CBuffer(m, n, n, True, init=c_init, extra_rows=1)
    got, raw = run_gemm_mxfp8(m, n, k, 1.0, A, SA, B, SB, 1.0, cbuf, workspace=ws)
    ref, bound = oracle.default().gemm_mxfp8(m, n, k, 1.0, A, SA, B, SB, 1.0, c_init)
    worst = assert_parity(got, ref, bound, 1.0, 1.0, c_input_values(c_init, True), True, "mxfp8 4096^2 x 2048")
    print(f"mxfp8 4096x4096x2048 beta=1 bf16: worst |err|/tol = {worst:.3g}")
    cbuf.assert_guard_intact(raw)


def test_mxfp8_alpha_zero_and_argument_errors():
    import blas3_tensor_core_gb300 as bm
    t = torch()
    m, n, k = 64, 64, 64
    C = t.full((m, n), 3.0, dtype=t.float32, device="cuda")
    h = t.cuda.current_stream().cuda_stream
    # alpha == 0: C = beta * C, operands and scales unread (null pointers allowed)
    assert bm.bm_gemm_mxfp8(m, n, k, 0.0, None, k, None, None, k, None, 0.5, C.data_ptr(), n, bm.BM_C_F32,
                            None, 0, h) == bm.BM_OK
    t.cuda.synchronize()
    assert bool(t.all(C == 1.5))
    buf = t.zeros(4096, dtype=t.uint8, device="cuda")
    base = buf.data_ptr()
    assert bm.bm_gemm_mxfp8(m, n, k, 1.0, base, k, None, base, k, base, 0.0, C.data_ptr(), n, bm.BM_C_F32,
                            None, 0, h) == bm.BM_ERR_INVALID_VALUE
    assert bm.bm_gemm_mxfp8(m, n, k, 1.0, base, k, base + 8, base, k, base, 0.0, C.data_ptr(), n, bm.BM_C_F32,
                            None, 0, h) == bm.BM_ERR_MISALIGNED
