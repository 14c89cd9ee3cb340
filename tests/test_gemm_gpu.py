"""GEMM parity: the CUDA path (through the C ABI) against the CPU oracle, on a GB300.

Small and ragged shapes are compared element by element on the whole output
(several tiles, ragged edges in m, n and k); the workloads at full size are
compared on every element in tests/test_full_size_gpu.py. Exact-integer inputs pin the descriptors and
the tensor-memory layout bit for bit; Gaussian inputs use the tolerance
1e-3 * |alpha| * sum|a*b| (+ 2^-8 |ref| for BF16 output).
"""

import itertools

import numpy as np
import pytest

import bm_inputs as gen
import oracle
from gpu_helpers import (VARIANT_IDS, VARIANTS, CBuffer, assert_parity, c_input_values, operand, run_gemm,
                         tile_samples, tile_variant, torch)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from blas3_tensor_core_gb300 import build
    build.build()
    assert torch().cuda.is_available()


def _stored(rows, cols, trans):
    return (cols, rows) if trans else (rows, cols)


def _pad_for(cols, elem_bytes):
    per = 16 // elem_bytes
    return (-cols) % per + per  # always pad: the gap must never be read


def _operands(m, n, k, ta, tb, dist, seed, std=1.0, lo=-1.0, hi=1.0):
    ra, ca = _stored(m, k, ta)
    rb, cb = _stored(k, n, tb)
    A = operand(ra, ca, dist, seed, std, lo, hi, pad=_pad_for(ca, 2))
    B = operand(rb, cb, dist, seed + 1, std, lo, hi, pad=_pad_for(cb, 2))
    return A, B


def _ldc(n, bf16):
    per = 8 if bf16 else 4
    return n + (-n) % per + per


ORC = None


def orc():
    global ORC
    if ORC is None:
        ORC = oracle.default()
    return ORC


# ----------------------------------------------------------------------------- exact
@pytest.mark.parametrize("variant", VARIANTS, ids=VARIANT_IDS)
@pytest.mark.parametrize("ta,tb", list(itertools.product((0, 1), (0, 1))))
@pytest.mark.parametrize("shape", [(256, 256, 256), (200, 300, 136), (129, 520, 64), (1, 8, 8), (520, 264, 72)])
def test_exact_integer_inputs_bitwise(shape, ta, tb, variant):
    m, n, k = shape
    A, B = _operands(m, n, k, ta, tb, "int", seed=11, lo=-8, hi=8)
    cbuf = CBuffer(m, n, _ldc(n, False), False, init=np.full((m, n), np.nan, np.float32))  # beta = 0: unread
    with tile_variant(variant):
        got, raw = run_gemm(m, n, k, ta, tb, 1.0, A, B, 0.0, cbuf)
    ref, _ = orc().gemm(m, n, k, ta, tb, 1.0, A, B)
    assert np.array_equal(got, ref), f"max |diff| {np.max(np.abs(got - ref))}"
    cbuf.assert_guard_intact(raw)


@pytest.mark.parametrize("variant", VARIANTS, ids=VARIANT_IDS)
def test_exact_integer_beta_accumulate_bitwise(variant):
    m, n, k = 384, 264, 200
    A, B = _operands(m, n, k, 0, 0, "int", seed=21, lo=-8, hi=8)
    c0 = gen.integers(23, m * n, -100, 100).reshape(m, n).astype(np.float32)
    cbuf = CBuffer(m, n, _ldc(n, False), False, init=c0)
    with tile_variant(variant):
        got, raw = run_gemm(m, n, k, 0, 0, 2.0, A, B, -1.0, cbuf)
    ref, _ = orc().gemm(m, n, k, 0, 0, 2.0, A, B, -1.0, c0)
    assert np.array_equal(got, ref)
    cbuf.assert_guard_intact(raw)


# ----------------------------------------------------------------------------- tolerance
def test_config_256_uniform_fp32():
    """256^3, A and B uniform in [-1, 1] rounded to bf16, FP32 C, alpha = 1, beta = 0."""
    m = n = k = 256
    A = operand(m, k, "uniform", seed=1)
    B = operand(k, n, "uniform", seed=2)
    cbuf = CBuffer(m, n, n, False, init=np.full((m, n), np.nan, np.float32))
    got, raw = run_gemm(m, n, k, 0, 0, 1.0, A, B, 0.0, cbuf)
    ref, bound = orc().gemm(m, n, k, 0, 0, 1.0, A, B)
    assert_parity(got, ref, bound, 1.0, 0.0, None, False, "256^3 fp32")
    cbuf.assert_guard_intact(raw)


@pytest.mark.parametrize("variant", [0, 3], ids=["auto", "pair256x256"])
@pytest.mark.parametrize("ta,tb", list(itertools.product((0, 1), (0, 1))))
@pytest.mark.parametrize("bf16_out,beta", [(False, 0.0), (False, 1.5), (True, 0.0), (True, -0.5)])
def test_gaussian_ragged_multi_tile(ta, tb, bf16_out, beta, variant):
    m, n, k = 640, 520, 328
    alpha = -0.75
    A, B = _operands(m, n, k, ta, tb, "normal", seed=31)
    c0 = gen.matrix_f32(m, n, "normal", seed=33)
    c_init = gen.f32_to_bf16_bits(c0) if bf16_out else c0
    cbuf = CBuffer(m, n, _ldc(n, bf16_out), bf16_out, init=c_init)
    with tile_variant(variant):
        got, raw = run_gemm(m, n, k, ta, tb, alpha, A, B, beta, cbuf)
    ref, bound = orc().gemm(m, n, k, ta, tb, alpha, A, B, beta, c_init if beta != 0 else None)
    assert_parity(got, ref, bound, alpha, beta, c_input_values(c_init, bf16_out), bf16_out, "ragged")
    cbuf.assert_guard_intact(raw)


def test_backward_shaped_small_transA_beta1_bf16():
    """dW += dY^T X in miniature: transA, K small, beta = 1 into an existing bf16 C, N(0, 0.02)."""
    m, n, k = 384, 640, 256
    A, B = _operands(m, n, k, 1, 0, "normal", seed=41, std=0.02)
    c_init = gen.matrix_bf16(m, n, "normal", seed=43, std=0.02)
    cbuf = CBuffer(m, n, _ldc(n, True), True, init=c_init)
    got, raw = run_gemm(m, n, k, 1, 0, 1.0, A, B, 1.0, cbuf)
    ref, bound = orc().gemm(m, n, k, 1, 0, 1.0, A, B, 1.0, c_init)
    assert_parity(got, ref, bound, 1.0, 1.0, c_input_values(c_init, True), True, "dW small")
    cbuf.assert_guard_intact(raw)


# ----------------------------------------------------------------------------- BLAS conventions
def test_alpha_zero_does_not_read_a_or_b():
    m, n, k = 130, 260, 70
    A = np.full((m, 72), gen.BF16_NAN, np.uint16)
    B = np.full((k, 264), gen.BF16_NAN, np.uint16)
    c0 = gen.matrix_f32(m, n, "normal", seed=51)
    cbuf = CBuffer(m, n, 264, False, init=c0)
    got, raw = run_gemm(m, n, k, 0, 0, 0.0, A, B, -2.0, cbuf)
    assert np.array_equal(got, (-2.0 * c0).astype(np.float32).astype(np.float64))
    cbuf.assert_guard_intact(raw)


def test_k_zero_gives_beta_c_and_beta_zero_gives_zero():
    m, n = 70, 36
    A = np.zeros((m, 8), np.uint16)
    B = np.zeros((8, 40), np.uint16)
    c0 = gen.matrix_bf16(m, n, "normal", seed=52)
    cbuf = CBuffer(m, n, 40, True, init=c0)
    got, raw = run_gemm(m, n, 0, 0, 0, 1.0, A, B, 0.5, cbuf)
    assert np.array_equal(got, 0.5 * gen.bf16_bits_to_f32(c0).astype(np.float64))
    cbuf.assert_guard_intact(raw)
    cbuf2 = CBuffer(m, n, 40, False, init=np.full((m, n), np.nan, np.float32))
    got, raw = run_gemm(m, n, 0, 0, 0, 1.0, A, B, 0.0, cbuf2)
    assert np.all(got == 0.0)
    cbuf2.assert_guard_intact(raw)


# ----------------------------------------------------------------------------- split K
@pytest.mark.parametrize("variant", [0, 3], ids=["auto", "pair256x256"])
def test_split_k_matches_oracle_and_is_deterministic(variant):
    import blas3_tensor_core_gb300 as bm
    t = torch()
    m, n, k = 512, 520, 8192
    A, B = _operands(m, n, k, 0, 0, "normal", seed=61)
    outs = []
    with tile_variant(variant):
        need = bm.bm_gemm_bf16_workspace_size(m, n, k)
        st, plan = bm.bm_gemm_bf16_plan(m, n, k, need)
        assert plan.k_splits > 1 and plan.cta_pair == (2 if variant == 3 else 1)
        ws = t.empty(need // 4 + 64, dtype=t.float32, device="cuda")
        for _ in range(2):
            cbuf = CBuffer(m, n, _ldc(n, False), False, init=np.full((m, n), np.nan, np.float32))
            got, raw = run_gemm(m, n, k, 0, 0, 1.0, A, B, 0.0, cbuf, workspace=ws)
            cbuf.assert_guard_intact(raw)
            outs.append(got)
    assert np.array_equal(outs[0], outs[1])
    rows, cols = tile_samples(m, n, per_tile=64, seed=3)
    ref, bound = orc().gemm_entries(k, 0, 0, 1.0, A, B, rows, cols)
    assert_parity(outs[0][rows, cols], ref, bound, 1.0, 0.0, None, False, "split-K")
    cbuf = CBuffer(m, n, _ldc(n, False), False)
    plain, _ = run_gemm(m, n, k, 0, 0, 1.0, A, B, 0.0, cbuf)  # no workspace: one split
    assert_parity(plain[rows, cols], ref, bound, 1.0, 0.0, None, False, "no split")


@pytest.mark.parametrize("variant", [0, 1, 2], ids=["auto", "single128x256", "single128x128"])
def test_tail_split_exact_and_deterministic(variant):
    """The tiles of a partly filled last wave are split along K over the idle SMs.

    Their units run first, and per 32-row region of a split tile the last unit to
    store its partial sums the slots and writes C inside the kernel. The region
    counters sit in the workspace after the slots and carry a per-launch tag, so
    the workspace may start with any bytes: it is filled with random bits here
    before the first call, and with a stale-looking pattern before the third.
    """
    import blas3_tensor_core_gb300 as bm
    t = torch()
    m, n, k = 2560, 2048, 3072  # SM pairs: 80 tiles = 76 + 4; single SMs: 160 tiles = 152 + 8
    A, B = _operands(m, n, k, 0, 0, "int", seed=81, lo=-8, hi=8)
    c0 = gen.integers(83, m * n, -100, 100).reshape(m, n).astype(np.float32)
    with tile_variant(variant):
        need = bm.bm_gemm_bf16_workspace_size(m, n, k)
        plan = bm.bm_gemm_bf16_plan(m, n, k, need)[1]
        assert plan.split_tiles > 0 and plan.k_splits > 1 and plan.kernels == 1
        ws = t.empty(need // 4, dtype=t.float32, device="cuda")
        g = t.Generator(device="cuda")
        g.manual_seed(5)
        ws.view(t.int32).copy_(t.randint(-2**31, 2**31 - 1, (need // 4,), dtype=t.int32, device="cuda", generator=g))
        slot_bytes = plan.k_splits * plan.split_tiles * plan.tile_m * plan.tile_n * 4
        assert need - slot_bytes == plan.split_tiles * plan.cta_pair * 8 * 8  # one counter per warp region
        outs = []
        for i in range(3):
            if i == 2:  # every counter as an earlier launch (tag 1) left it after one arrival
                ws.view(t.int64)[slot_bytes // 8:].fill_((1 << 16) | 1)
            cbuf = CBuffer(m, n, n, False, init=c0)
            got, raw = run_gemm(m, n, k, 0, 0, 1.0, A, B, -1.0, cbuf, workspace=ws)
            cbuf.assert_guard_intact(raw)
            outs.append(got)
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])
    ref, _ = orc().gemm(m, n, k, 0, 0, 1.0, A, B, -1.0, c0)
    assert np.array_equal(outs[0], ref)


@pytest.mark.parametrize("beta", [0.0, 1.0], ids=["beta0", "beta1"])
def test_tail_split_depends_on_beta(beta):
    """4096^2 x 2048: the 28 tiles of the last wave save 4.1 us of mainloop by a 2-way K split.
    That pays when the split tiles need no combine with C (beta == 0, split and summed in the
    kernel) and not otherwise (beta != 0, whole tiles). Either plan must give the exact result:
    small integers, checked on every row of four columns through the split tiles (the last two
    tile columns) and on samples everywhere else."""
    import blas3_tensor_core_gb300 as bm
    t = torch()
    m = n = 4096
    k = 2048
    st, plan = bm.bm_gemm_bf16_plan(m, n, k, bm.bm_gemm_bf16_workspace_size(m, n, k))
    assert (plan.split_tiles, plan.k_splits, plan.kernels) == (28, 2, 1)   # the plan reported is beta == 0's
    A, B = _operands(m, n, k, 0, 0, "int", seed=87, lo=-2, hi=2)
    c0 = gen.integers(88, m * n, -30, 30).reshape(m, n).astype(np.float32)
    need = bm.bm_gemm_bf16_workspace_size(m, n, k)
    ws = t.empty(need // 4, dtype=t.float32, device="cuda")
    cbuf = CBuffer(m, n, n, False, init=c0)
    got, raw = run_gemm(m, n, k, 0, 0, 1.0, A, B, beta, cbuf, workspace=ws)
    cbuf.assert_guard_intact(raw)
    cols_full = np.array([3584, 3700, 3840, 4095])
    band_r = np.tile(np.arange(m), cols_full.size)
    band_c = np.repeat(cols_full, m)
    rows, cols = tile_samples(m, n, tile_m=256, tile_n=256, per_tile=8, seed=14, extra=(band_r, band_c))
    ref, _ = orc().gemm_entries(k, 0, 0, 1.0, A, B, rows, cols, beta, c0 if beta != 0 else None)
    assert np.array_equal(got[rows, cols], ref)


def test_tail_split_ragged_many_splits_bf16_beta():
    """Ragged m, n and k; the 4 tail tiles split 10 ways and summed in the kernel, into bf16 C with beta."""
    import blas3_tensor_core_gb300 as bm
    t = torch()
    m, n, k = 2500, 2000, 3000  # 10 x 8 pair tiles = 76 + 4
    alpha, beta = 0.75, 0.5
    A, B = _operands(m, n, k, 0, 0, "normal", seed=85)
    c_init = gen.matrix_bf16(m, n, "normal", seed=86)
    need = bm.bm_gemm_bf16_workspace_size(m, n, k)
    plan = bm.bm_gemm_bf16_plan(m, n, k, need)[1]
    assert (plan.split_tiles, plan.k_splits, plan.kernels) == (4, 10, 1)
    ws = t.full((need // 4,), float("nan"), dtype=t.float32, device="cuda")
    cbuf = CBuffer(m, n, _ldc(n, True), True, init=c_init)
    got, raw = run_gemm(m, n, k, 0, 0, alpha, A, B, beta, cbuf, workspace=ws)
    cbuf.assert_guard_intact(raw)
    band_r = np.repeat(np.arange(1280, m), 256)  # the split tiles: last tile column, last 4 tile rows
    band_c = np.tile(np.arange(n - 256, n), m - 1280)
    rows, cols = tile_samples(m, n, per_tile=8, seed=13, extra=(band_r, band_c))
    ref, bound = orc().gemm_entries(k, 0, 0, alpha, A, B, rows, cols, beta, c_init)
    assert_parity(got[rows, cols], ref, bound, alpha, beta, c_input_values(c_init, True)[rows, cols], True,
                  "tail split x10")


@pytest.mark.parametrize("m,n,k,ta,tb", [(2560, 2048, 1024, 0, 0), (2560, 2048, 512, 0, 1), (2560, 2048, 1024, 1, 0),
                                         (2500, 1976, 1000, 0, 0)],
                         ids=["nn", "nt_k512", "tn", "ragged"])
@pytest.mark.parametrize("beta", [0.0, -1.0])
@pytest.mark.parametrize("bf16_out", [False, True])
def test_n_half_tail_whole_output_exact(m, n, k, ta, tb, beta, bf16_out):
    """80 pair tiles = 76 + 4 with too few k-blocks for a K split: each of the 4 tail tiles
    runs as two units of half its columns (MMA N = 128 over half of each CTA's B rows), on
    8 SM pairs, with no partial sums. Small integers make every element exact, so the whole
    output (and the guard band) is compared with the oracle; the ragged shape puts part of
    the last tile column's halves outside n."""
    import blas3_tensor_core_gb300 as bm
    p = bm.bm_gemm_bf16_plan(m, n, k, 0)[1]
    assert (p.split_tiles, p.k_splits, p.n_splits) == (4, 1, 2)
    A, B = _operands(m, n, k, ta, tb, "int", seed=95, lo=-3, hi=3)
    c0 = gen.integers(96, m * n, -30, 30).reshape(m, n).astype(np.float32)
    c_init = gen.f32_to_bf16_bits(c0) if bf16_out else c0
    cbuf = CBuffer(m, n, _ldc(n, bf16_out), bf16_out, init=c_init)
    got, raw = run_gemm(m, n, k, ta, tb, 1.0, A, B, beta, cbuf)
    cbuf.assert_guard_intact(raw)
    ref, _ = orc().gemm(m, n, k, ta, tb, 1.0, A, B, beta, c_init if beta != 0.0 else None)
    if bf16_out:
        ref = gen.bf16_bits_to_f32(gen.f32_to_bf16_bits(ref.astype(np.float32))).astype(np.float64)
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("m,n,k,beta,bf16_out,ws", [
    (2600, 2602, 512, 0.0, False, False),    # 121 whole pair tiles, TMA-store path when aligned
    (2600, 2605, 512, -1.0, True, False),    # the same, group path when aligned
    (2225, 2162, 2464, 0.0, False, True),    # 81 pair tiles, the last 5 split 8 ways along K
    (2225, 2163, 2048, -1.0, True, True),
    (2219, 2162, 569, -1.0, False, False),   # tail tiles planned as N halves, run whole
    (700, 1029, 320, 0.0, True, False),      # short K: 128 x 256 tiles on single SMs
], ids=["pair_f32", "pair_bf16_beta", "tail_k_f32", "tail_k_bf16_beta", "n_half_f32_beta", "single_bf16"])
def test_row_end_off_16_bytes_leaves_columns_past_n_intact(m, n, k, beta, bf16_out, ws):
    """A row of C that does not end on a 16-byte boundary (fp32 n = 4q + 2 or 3, bf16 n = 8q + 5):
    a tiled TMA store would also write the columns from n to the next boundary, so these calls
    store C with masked plain stores. Small integers: the whole output equals the oracle bit
    for bit, and the columns past n (inside ldc) and the rows below C keep their canaries."""
    import blas3_tensor_core_gb300 as bm
    t = torch()
    A, B = _operands(m, n, k, 0, 1, "int", seed=97, lo=-3, hi=3)
    c0 = gen.integers(98, m * n, -30, 30).reshape(m, n).astype(np.float32)
    c_init = gen.f32_to_bf16_bits(c0) if bf16_out else c0
    cbuf = CBuffer(m, n, _ldc(n, bf16_out), bf16_out, init=c_init)
    workspace = None
    if ws:
        need = bm.bm_gemm_bf16_workspace_size(m, n, k)
        assert bm.bm_gemm_bf16_plan(m, n, k, need)[1].k_splits > 1
        workspace = t.full((need // 4,), float("nan"), dtype=t.float32, device="cuda")
    got, raw = run_gemm(m, n, k, 0, 1, 1.0, A, B, beta, cbuf, workspace=workspace)
    cbuf.assert_guard_intact(raw)
    ref, _ = orc().gemm(m, n, k, 0, 1, 1.0, A, B, beta, c_init if beta != 0.0 else None)
    if bf16_out:
        ref = gen.bf16_bits_to_f32(gen.f32_to_bf16_bits(ref.astype(np.float32))).astype(np.float64)
    assert np.array_equal(got, ref)


def test_beta_tail_split_then_whole_tiles_whole_output_exact():
    """beta != 0 with a tail split summed in the kernel: 2560 x 2048 x 3072 has 80 pair
    tiles = 76 + 4, and the 4 are split 12 ways. The 48 split units go first (transposing
    path, partials, in-kernel sum) and their SM pairs then run whole tiles through the
    group path (TMA load of C, combine, store), whose first C chunk is loaded early only
    when the half's staging block is free. Small integers make every element exact, so
    the whole output is compared with the oracle bit for bit."""
    import blas3_tensor_core_gb300 as bm
    t = torch()
    m, n, k = 2560, 2048, 3072
    need = bm.bm_gemm_bf16_workspace_size(m, n, k)
    A, B = _operands(m, n, k, 0, 0, "int", seed=91, lo=-2, hi=2)
    c0 = gen.integers(92, m * n, -30, 30).reshape(m, n).astype(np.float32)
    ws = t.full((need // 4,), float("nan"), dtype=t.float32, device="cuda")
    cbuf = CBuffer(m, n, n + 4, False, init=c0)
    got, raw = run_gemm(m, n, k, 0, 0, 1.0, A, B, -1.0, cbuf, workspace=ws)
    cbuf.assert_guard_intact(raw)
    ref, _ = orc().gemm(m, n, k, 0, 0, 1.0, A, B, -1.0, c0)
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("bf16_out", [False, True])
def test_tail_split_graph_replays(bf16_out):
    """A CUDA graph replays its calls with the tags they were captured with; the
    last unit of each region resets its counter, so every replay starts clean.
    New inputs are copied into the captured buffers before each replay."""
    import blas3_tensor_core_gb300 as bm
    from gpu_helpers import bf16_to_device, device_to_numpy
    t = torch()
    m, n, k = 2560, 2048, 3072  # 80 pair tiles = 76 + 4; the 4 are split
    need = bm.bm_gemm_bf16_workspace_size(m, n, k)
    assert bm.bm_gemm_bf16_plan(m, n, k, need)[1].kernels == 1
    ws = t.zeros(need // 4, dtype=t.float32, device="cuda")
    dA = t.empty((m, k), dtype=t.bfloat16, device="cuda")
    dB = t.empty((k, n), dtype=t.bfloat16, device="cuda")
    dC = t.empty((m, n), dtype=t.bfloat16 if bf16_out else t.float32, device="cuda")
    ct = bm.BM_C_BF16 if bf16_out else bm.BM_C_F32

    def call(h):
        assert bm.bm_gemm_bf16(m, n, k, 0, 0, 1.0, dA.data_ptr(), k, dB.data_ptr(), n, 0.0, dC.data_ptr(), n, ct,
                               ws.data_ptr(), need, h) == bm.BM_OK

    side = t.cuda.Stream()
    side.wait_stream(t.cuda.current_stream())
    with t.cuda.stream(side):
        call(side.cuda_stream)  # first-call set-up outside the capture
    t.cuda.current_stream().wait_stream(side)
    t.cuda.synchronize()
    graph = t.cuda.CUDAGraph()
    with t.cuda.graph(graph):
        call(t.cuda.current_stream().cuda_stream)
    # the split tiles are the last ones of the raster: the last tile column, lower rows;
    # all of the last 256 columns, and samples elsewhere
    band_r = np.repeat(np.arange(m), 256)
    band_c = np.tile(np.arange(n - 256, n), m)
    rows, cols = tile_samples(m, n, per_tile=24, seed=12, extra=(band_r, band_c))
    for rep in range(3):
        A = operand(m, k, "int", 100 + rep, lo=-4, hi=4)
        B = operand(k, n, "int", 200 + rep, lo=-4, hi=4)
        dA.copy_(bf16_to_device(A))
        dB.copy_(bf16_to_device(B))
        graph.replay()
        t.cuda.synchronize()
        assert bm.bm_get_last_device_error(t.cuda.current_stream().cuda_stream) == bm.BM_OK
        got = (gen.bf16_bits_to_f32(device_to_numpy(dC)) if bf16_out else dC.cpu().numpy()).astype(np.float64)
        ref, _ = orc().gemm_entries(k, 0, 0, 1.0, A, B, rows, cols)
        if bf16_out:
            ref = gen.bf16_bits_to_f32(gen.f32_to_bf16_bits(ref.astype(np.float32))).astype(np.float64)
        assert np.array_equal(got[rows, cols], ref), f"replay {rep}"
    del graph


# ----------------------------------------------------------------------------- stream ordering
@pytest.mark.parametrize("m,n,k", [(2048, 2048, 1024), (512, 512, 8192)], ids=["pair_tiles", "split_k"])
def test_dependent_calls_back_to_back(m, n, k):
    """D = A B; D = 2 D (alpha = 0 path); E = D B2 -- queued with no host synchronisation.

    Each kernel starts its set-up while the previous one finishes (programmatic
    dependent launch) and must still see the previous kernel's complete output.
    """
    import blas3_tensor_core_gb300 as bm
    from gpu_helpers import bf16_to_device, device_to_numpy
    t = torch()
    A = operand(m, k, "int", 91, lo=-4, hi=4)
    B = operand(k, n, "int", 92, lo=-4, hi=4)
    B2 = operand(n, n, "int", 93, lo=-2, hi=2)
    dA, dB, dB2 = bf16_to_device(A), bf16_to_device(B), bf16_to_device(B2)
    dD = t.empty((m, n), dtype=t.float32, device="cuda")
    dE = t.empty((m, n), dtype=t.float32, device="cuda")
    need = max(bm.bm_gemm_bf16_workspace_size(m, n, k), bm.bm_gemm_bf16_workspace_size(m, n, n))
    ws = t.empty(max(need // 4, 64), dtype=t.float32, device="cuda")
    dDb = t.empty((m, n), dtype=t.bfloat16, device="cuda")
    h = t.cuda.current_stream().cuda_stream
    assert bm.bm_gemm_bf16(m, n, k, 0, 0, 1.0, dA.data_ptr(), k, dB.data_ptr(), n, 0.0, dD.data_ptr(), n,
                           bm.BM_C_F32, ws.data_ptr(), need, h) == bm.BM_OK
    assert bm.bm_gemm_bf16(m, n, k, 0, 0, 0.0, None, k, None, n, 2.0, dD.data_ptr(), n,
                           bm.BM_C_F32, None, 0, h) == bm.BM_OK
    # bf16 copy of D on the same stream (a torch kernel between two of ours)
    dDb.copy_(dD)
    assert bm.bm_gemm_bf16(m, n, n, 0, 0, 1.0, dDb.data_ptr(), n, dB2.data_ptr(), n, 0.0, dE.data_ptr(), n,
                           bm.BM_C_F32, ws.data_ptr(), need, h) == bm.BM_OK
    t.cuda.synchronize()
    assert bm.bm_get_last_device_error(h) == bm.BM_OK
    D = dD.cpu().numpy().astype(np.float64)
    Db = device_to_numpy(dDb)
    E = dE.cpu().numpy().astype(np.float64)
    rows, cols = tile_samples(m, n, per_tile=8, seed=9)
    refD, _ = orc().gemm_entries(k, 0, 0, 2.0, A, B, rows, cols)
    assert np.array_equal(D[rows, cols], refD)  # small integers: exact
    refE, boundE = orc().gemm_entries(n, 0, 0, 1.0, Db, B2, rows, cols)
    assert_parity(E[rows, cols], refE, boundE, 1.0, 0.0, None, False, "E = D B2")


# ----------------------------------------------------------------------------- persistence
@pytest.mark.parametrize("variant", [0, 1], ids=["auto", "single128x256"])
def test_persistent_many_tiles_exact(variant):
    """More tiles than SMs (each CTA loops over several tiles and both accumulators)."""
    m, n, k = 4096, 2048, 192
    A, B = _operands(m, n, k, 0, 0, "int", seed=71, lo=-8, hi=8)
    cbuf = CBuffer(m, n, n, False)
    with tile_variant(variant):
        got, raw = run_gemm(m, n, k, 0, 0, 1.0, A, B, 0.0, cbuf)
    rows, cols = tile_samples(m, n, per_tile=16, seed=4)
    ref, _ = orc().gemm_entries(k, 0, 0, 1.0, A, B, rows, cols)
    assert np.array_equal(got[rows, cols], ref)
    # whole rows, one per tile row, exactly
    rr = np.arange(0, m, 128) + 37
    full_rows = np.repeat(rr, n)
    full_cols = np.tile(np.arange(n), len(rr))
    ref_rows, _ = orc().gemm_entries(k, 0, 0, 1.0, A, B, full_rows, full_cols)
    assert np.array_equal(got[full_rows, full_cols], ref_rows)
    cbuf.assert_guard_intact(raw)


@pytest.mark.parametrize("variant", [0, 3], ids=["auto", "pair256x256"])
@pytest.mark.parametrize("beta,bf16_out", [(0.0, True), (-1.0, False)], ids=["beta0_bf16", "beta-1_f32"])
def test_every_tile_split_exact_and_replayed(variant, beta, bf16_out):
    """512 x 512 x 8192: too few tiles for the GPU, so every tile is split along K and a
    second kernel sums the partials. The workspace holds random bits before the first call;
    a CUDA graph of the call is then replayed three times with new inputs. Small integers
    make every result exact, into bf16 C with beta = 0 and FP32 C with beta = -1."""
    import blas3_tensor_core_gb300 as bm
    from gpu_helpers import bf16_to_device, device_to_numpy
    t = torch()
    m, n, k = 512, 512, 8192
    with tile_variant(variant):
        need = bm.bm_gemm_bf16_workspace_size(m, n, k)
        plan = bm.bm_gemm_bf16_plan(m, n, k, need)[1]
        assert plan.split_tiles == plan.tiles and plan.k_splits > 1 and plan.kernels == 2
        assert need == plan.k_splits * plan.tiles * plan.tile_m * plan.tile_n * 4
        ws = t.empty((need // 4,), dtype=t.float32, device="cuda")
        g = t.Generator(device="cuda")
        g.manual_seed(7)
        ws.view(t.int32).copy_(t.randint(-2**31, 2**31 - 1, (need // 4,), dtype=t.int32, device="cuda", generator=g))
        dA = t.empty((m, k), dtype=t.bfloat16, device="cuda")
        dB = t.empty((k, n), dtype=t.bfloat16, device="cuda")
        dC = t.empty((m, n), dtype=t.bfloat16 if bf16_out else t.float32, device="cuda")
        ct = bm.BM_C_BF16 if bf16_out else bm.BM_C_F32

        def call(h):
            assert bm.bm_gemm_bf16(m, n, k, 0, 0, 1.0, dA.data_ptr(), k, dB.data_ptr(), n, beta, dC.data_ptr(), n,
                                   ct, ws.data_ptr(), need, h) == bm.BM_OK

        def check(seed):
            A = operand(m, k, "int", seed, lo=-4, hi=4)
            B = operand(k, n, "int", seed + 1, lo=-4, hi=4)
            c0 = gen.integers(seed + 2, m * n, -40, 40).reshape(m, n).astype(np.float32)
            dA.copy_(bf16_to_device(A))
            dB.copy_(bf16_to_device(B))
            dC.copy_(t.from_numpy(c0).cuda().to(dC.dtype))
            return A, B, c0

        def compare(A, B, c0, what):
            got = (gen.bf16_bits_to_f32(device_to_numpy(dC)) if bf16_out else dC.cpu().numpy()).astype(np.float64)
            ref, _ = orc().gemm(m, n, k, 0, 0, 1.0, A, B, beta, c0 if beta != 0 else None)
            if bf16_out:
                ref = gen.bf16_bits_to_f32(gen.f32_to_bf16_bits(ref.astype(np.float32))).astype(np.float64)
            assert np.array_equal(got, ref), what

        h = t.cuda.current_stream().cuda_stream
        for rep in range(2):
            A, B, c0 = check(300 + rep)
            call(h)
            t.cuda.synchronize()
            assert bm.bm_get_last_device_error(h) == bm.BM_OK
            compare(A, B, c0, f"eager call {rep}")
        side = t.cuda.Stream()
        side.wait_stream(t.cuda.current_stream())
        with t.cuda.stream(side):
            call(side.cuda_stream)
        t.cuda.current_stream().wait_stream(side)
        t.cuda.synchronize()
        graph = t.cuda.CUDAGraph()
        with t.cuda.graph(graph):
            call(t.cuda.current_stream().cuda_stream)
        for rep in range(3):
            A, B, c0 = check(400 + rep)
            graph.replay()
            t.cuda.synchronize()
            assert bm.bm_get_last_device_error(h) == bm.BM_OK
            compare(A, B, c0, f"graph replay {rep}")
        del graph
