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

# automatic choice, 128 x 128 tiles on single SMs, 256 x 128 and 256 x 256 tiles on SM pairs
MX_VARIANTS = [0, 1, 2, 3]
MX_IDS = ["auto", "single128x128", "pair256x128", "pair256x256"]


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


@pytest.mark.parametrize("variant", [0, 2, 3], ids=["auto", "pair256x128", "pair256x256"])
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


@pytest.mark.parametrize("variant", [0, 2], ids=["auto", "pair256x128"])
def test_mxfp8_tail_split_beta_bf16(variant):
    """4096 x 4096 x 2048 on SM pairs (256 tiles of 256 x 256 = 3 waves of 76 + 28, or 512 of
    256 x 128 = 6 waves + 56); whole-output parity with beta into a bf16 C."""
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
    with tile_variant(variant):
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


# ----------------------------------------------------------------------------- quantization
def _quantize_on_gpu(X, rows, k, ldq):
    """bm_quantize_mxfp8 on bf16 bits X [rows, ldx]; returns (Q [rows, ldq] bytes, tiled S bytes)."""
    import blas3_tensor_core_gb300 as bm
    from gpu_helpers import bf16_to_device, u8_to_device
    t = torch()
    dX = bf16_to_device(X)
    dQ = u8_to_device(np.full((rows, ldq), 0xA5, np.uint8))           # sentinel past column k
    dS = u8_to_device(np.full(bm.mxfp8_scale_bytes(rows, k), 0xEE, np.uint8))
    st = bm.bm_quantize_mxfp8(rows, k, dX.data_ptr(), X.shape[1], dQ.data_ptr(), ldq, dS.data_ptr(),
                              t.cuda.current_stream().cuda_stream)
    assert st == bm.BM_OK, bm.bm_status_string(st)
    t.cuda.synchronize()
    assert bm.bm_get_last_device_error(t.cuda.current_stream().cuda_stream) == bm.BM_OK
    return dQ.cpu().numpy(), dS.cpu().numpy()


def _check_quantized(X, rows, k, ldq, Qg, Sg):
    from gpu_helpers import mxfp8_tiled_scales
    Q, S = oracle.default().quantize_mxfp8(X, k)
    assert np.array_equal(Qg[:, :k], Q), f"{np.count_nonzero(Qg[:, :k] != Q)} E4M3 codes differ"
    assert np.all(Qg[:, k:] == 0xA5), "bytes past column k were written"
    assert np.array_equal(Sg, mxfp8_tiled_scales(S, rows, k, pad_code=0)), "scale codes or padding differ"
    return Q, S


def test_quantize_ragged_with_special_groups_bitwise():
    """300 x 200 (the last group of each row holds 8 elements), padded rows of NaN that must not be
    read, and planted groups: all zeros, a NaN, an infinity, values tiny enough to clamp the scale
    to 2^-127, values that saturate, and exact ties between E4M3 neighbours."""
    rows, k, ldx, ldq = 300, 200, 216, 224
    vals = gen.matrix_f32(rows, k, "normal", seed=81, std=2.0)
    vals[3, 32:64] = 0.0
    vals[4, 70] = np.nan
    vals[5, 10] = -np.inf
    vals[6] *= np.float32(2e-38)
    vals[7, 64:68] = [256.0, 8.5, 9.5, 17.0]
    vals[8, 0:3] = [500.0, -464.0, 448.0]
    vals[9, 192:200] = [1e-3, -2.0, 0.0, 0.5, 0.25, -0.125, 3.0, 1.0]
    X = gen.pad_ld(gen.f32_to_bf16_bits(vals), ldx, gen.BF16_NAN)
    Qg, Sg = _quantize_on_gpu(X, rows, k, ldq)
    Q, S = _check_quantized(X, rows, k, ldq, Qg, Sg)
    assert S[3, 1] == 0 and S[4, 2] == 255 and S[5, 0] == 255 and np.all(S[6] == 0)


@pytest.mark.parametrize("rows,k", [(1, 32), (128, 128), (129, 96), (4096, 4096)])
def test_quantize_shapes_bitwise(rows, k):
    X = gen.matrix_bf16(rows, k, "normal", seed=91)
    Qg, Sg = _quantize_on_gpu(X, rows, k, k + (-k) % 16)
    _check_quantized(X, rows, k, k + (-k) % 16, Qg, Sg)


def test_quantize_then_block_scaled_gemm():
    """The MXFP8 path end to end on the GPU: quantize BF16 A [m, k] and W [n, k], then C = A W^T
    from the codes and scales; the codes and scales equal the oracle's bit for bit, and C matches
    the oracle's block-scaled GEMM on them."""
    import blas3_tensor_core_gb300 as bm
    from gpu_helpers import bf16_to_device
    t = torch()
    m, n, k = 520, 264, 392
    A = gen.matrix_bf16(m, k, "normal", seed=101)
    W = gen.matrix_bf16(n, k, "normal", seed=102, std=0.05)
    h = t.cuda.current_stream().cuda_stream
    ldq = k + (-k) % 16
    dA, dW = bf16_to_device(A), bf16_to_device(W)
    dQa = t.empty((m, ldq), dtype=t.uint8, device="cuda")
    dQw = t.empty((n, ldq), dtype=t.uint8, device="cuda")
    dSa = t.empty(bm.mxfp8_scale_bytes(m, k), dtype=t.uint8, device="cuda")
    dSw = t.empty(bm.mxfp8_scale_bytes(n, k), dtype=t.uint8, device="cuda")
    assert bm.bm_quantize_mxfp8(m, k, dA.data_ptr(), k, dQa.data_ptr(), ldq, dSa.data_ptr(), h) == bm.BM_OK
    assert bm.bm_quantize_mxfp8(n, k, dW.data_ptr(), k, dQw.data_ptr(), ldq, dSw.data_ptr(), h) == bm.BM_OK
    cbuf = CBuffer(m, n, _ldc(n, True), True, init=np.zeros((m, n), np.uint16))
    assert bm.bm_gemm_mxfp8(m, n, k, 1.0, dQa.data_ptr(), ldq, dSa.data_ptr(), dQw.data_ptr(), ldq, dSw.data_ptr(),
                            0.0, cbuf.ptr, cbuf.ldc, bm.BM_C_BF16, None, 0, h) == bm.BM_OK
    t.cuda.synchronize()
    assert bm.bm_get_last_device_error(h) == bm.BM_OK
    Qa, Sa = oracle.default().quantize_mxfp8(A)
    Qw, Sw = oracle.default().quantize_mxfp8(W)
    assert np.array_equal(dQa.cpu().numpy()[:, :k], Qa) and np.array_equal(dQw.cpu().numpy()[:, :k], Qw)
    got, raw = cbuf.result()
    ref, bound = oracle.default().gemm_mxfp8(m, n, k, 1.0, Qa, Sa, Qw, Sw)
    assert_parity(got, ref, bound, 1.0, 0.0, None, True, "quantize + mxfp8 gemm")
    cbuf.assert_guard_intact(raw)


@pytest.mark.parametrize("m,n,k,bf16_out,beta", [(520, 262, 192, False, 0.0), (2304, 2306, 256, True, -1.0)],
                         ids=["single_f32", "pair_bf16_beta"])
def test_mxfp8_row_end_off_16_bytes_exact(m, n, k, bf16_out, beta):
    """Rows of C that do not end on a 16-byte boundary are stored with masked plain stores
    (a TMA store would also write the columns from n to the boundary). Exact data (scales 2^-1
    .. 2^1): the whole output equals the oracle, and the columns past n and the rows below C
    are unchanged."""
    A = _codes(m, k, "int", 31)
    B = _codes(n, k, "int", 32)
    SA = _scales(m, k, 33, 126, 128)
    SB = _scales(n, k, 34, 126, 128)
    c0 = gen.integers(35, m * n, -30, 30).reshape(m, n).astype(np.float32)
    c_init = gen.f32_to_bf16_bits(c0) if bf16_out else c0
    cbuf = CBuffer(m, n, _ldc(n, bf16_out), bf16_out, init=c_init)
    got, raw = run_gemm_mxfp8(m, n, k, 1.0, A, SA, B, SB, beta, cbuf)
    cbuf.assert_guard_intact(raw)
    ref, _ = oracle.default().gemm_mxfp8(m, n, k, 1.0, A, SA, B, SB, beta, c_init if beta != 0 else None)
    if bf16_out:
        ref = gen.bf16_bits_to_f32(gen.f32_to_bf16_bits(ref.astype(np.float32))).astype(np.float64)
    assert np.array_equal(got, ref), _explain(got, ref)
