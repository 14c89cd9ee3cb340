"""The GEMM entry point that allocates nothing, bm_gemm_bf16_noalloc, on a GB300.

Some callers cannot call cudaMalloc: a framework that owns all device memory
through its own pool, a plug-in called back by another library without an
allocator, or a latency-critical path that cannot afford cudaMalloc's implicit
synchronisation. For them the library keeps its split-K scratch in a static
device array. These tests call that entry point through the C ABI and compare
it with bm_gemm_bf16 given a caller-owned workspace, on two calls in a row
(the array keeps the previous call's contents), and check that a shape whose
partial sums do not fit the array is refused without touching C.

The file name sorts last so that a run that stops at the first failure has
already run every other test. It depends on no state left by other tests.
"""

import numpy as np
import pytest

import bm_inputs as gen
import oracle
from gpu_helpers import CBuffer, bf16_to_device, operand, torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from blas3_tensor_core_gb300 import build
    build.build()
    assert torch().cuda.is_available()


def _bound(A, B):
    a = gen.bf16_bits_to_f32(A).astype(np.float64)
    b = gen.bf16_bits_to_f32(B).astype(np.float64)
    return np.abs(a) @ np.abs(b)


def _with_workspace(m, n, k, dA, dB, lda, ldb, alpha, beta, c_init, bf16):
    """The existing entry point, with a workspace of the size it asks for."""
    import blas3_tensor_core_gb300 as bm
    t = torch()
    need = bm.bm_gemm_bf16_workspace_size(m, n, k)
    ws = t.empty(max(need // 4, 64), dtype=t.float32, device="cuda")
    cbuf = CBuffer(m, n, n, bf16, init=c_init)
    st = bm.bm_gemm_bf16(m, n, k, 0, 0, alpha, dA.data_ptr(), lda, dB.data_ptr(), ldb, beta, cbuf.ptr, n,
                         bm.BM_C_BF16 if bf16 else bm.BM_C_F32, ws.data_ptr(), need,
                         t.cuda.current_stream().cuda_stream)
    assert st == bm.BM_OK
    t.cuda.synchronize()
    return cbuf.result()[0], need


def _noalloc(m, n, k, dA, dB, lda, ldb, alpha, beta, c_init, bf16):
    import blas3_tensor_core_gb300 as bm
    t = torch()
    cbuf = CBuffer(m, n, n, bf16, init=c_init)
    st = bm.bm_gemm_bf16_noalloc(m, n, k, 0, 0, alpha, dA.data_ptr(), lda, dB.data_ptr(), ldb, beta, cbuf.ptr,
                                 n, bm.BM_C_BF16 if bf16 else bm.BM_C_F32, t.cuda.current_stream().cuda_stream)
    assert st == bm.BM_OK, bm.bm_status_string(st)
    t.cuda.synchronize()
    got, raw = cbuf.result()
    cbuf.assert_guard_intact(raw)
    return got


def test_split_k_without_allocation_matches_workspace_path_twice():
    import blas3_tensor_core_gb300 as bm
    m, n, k = 512, 520, 2048
    st, plan = bm.bm_gemm_bf16_plan(m, n, k, bm.bm_gemm_bf16_workspace_size(m, n, k))
    assert plan.k_splits > 1 and plan.workspace_bytes <= bm.BM_NOALLOC_SCRATCH_BYTES
    # two calls in a row, on different inputs: the second must not see the first's partials
    for seed in (11, 21):
        A = operand(m, k, "normal", seed)
        B = operand(k, n, "normal", seed + 1)
        dA, dB = bf16_to_device(A), bf16_to_device(B)
        want, _ = _with_workspace(m, n, k, dA, dB, k, n, 1.0, 0.0, None, True)
        got = _noalloc(m, n, k, dA, dB, k, n, 1.0, 0.0, None, True)
        ok, worst, where = oracle.compare(got, want, _bound(A, B), 1.0, 0.0, None, True)
        assert ok, (seed, worst, where)


def test_tail_split_summed_in_kernel_without_allocation_three_times():
    """Tail tiles split along K and summed inside the kernel: the partial slots and the
    region counters both live in the static array. Three calls in a row on different
    integer inputs (the counters are reset by each call's last units), with beta = 0
    and beta = -1; small integers make every result exact, so the two entry points
    must agree bit for bit."""
    import blas3_tensor_core_gb300 as bm
    m, n, k = 2560, 2048, 3072
    st, plan = bm.bm_gemm_bf16_plan(m, n, k, bm.bm_gemm_bf16_workspace_size(m, n, k))
    assert plan.split_tiles > 0 and plan.k_splits > 1 and plan.kernels == 1
    assert plan.workspace_bytes <= bm.BM_NOALLOC_SCRATCH_BYTES
    for seed, beta in ((61, 0.0), (71, -1.0), (81, 0.0)):
        A = operand(m, k, "int", seed, lo=-4, hi=4)
        B = operand(k, n, "int", seed + 1, lo=-4, hi=4)
        c0 = gen.integers(seed + 2, m * n, -50, 50).reshape(m, n).astype(np.float32)
        dA, dB = bf16_to_device(A), bf16_to_device(B)
        want, _ = _with_workspace(m, n, k, dA, dB, k, n, 1.0, beta, c0, False)
        got = _noalloc(m, n, k, dA, dB, k, n, 1.0, beta, c0, False)
        assert np.array_equal(got, want), seed


def test_without_split_and_with_beta():
    m, n, k = 256, 264, 256
    A = operand(m, k, "normal", 31)
    B = operand(k, n, "normal", 32)
    c0 = gen.matrix_f32(m, n, "normal", seed=33)
    dA, dB = bf16_to_device(A), bf16_to_device(B)
    want, need = _with_workspace(m, n, k, dA, dB, k, n, -0.5, 1.5, c0, False)
    for _ in range(2):
        got = _noalloc(m, n, k, dA, dB, k, n, -0.5, 1.5, c0, False)
        ok, worst, _ = oracle.compare(got, want, _bound(A, B), -0.5, 1.5, c0.astype(np.float64), False)
        assert ok, worst


def test_plan_beyond_the_scratch_array_is_refused():
    import blas3_tensor_core_gb300 as bm
    t = torch()
    m, n, k = 512, 512, 8192
    assert bm.bm_gemm_bf16_workspace_size(m, n, k) > bm.BM_NOALLOC_SCRATCH_BYTES
    A = operand(m, k, "normal", 41)
    B = operand(k, n, "normal", 42)
    dA, dB = bf16_to_device(A), bf16_to_device(B)
    cbuf = CBuffer(m, n, n, True, init=np.zeros((m, n), np.uint16))
    st = bm.bm_gemm_bf16_noalloc(m, n, k, 0, 0, 1.0, dA.data_ptr(), k, dB.data_ptr(), n, 0.0, cbuf.ptr, n,
                                 bm.BM_C_BF16, t.cuda.current_stream().cuda_stream)
    assert st == bm.BM_ERR_WORKSPACE
    t.cuda.synchronize()
    _, raw = cbuf.result()
    assert np.array_equal(raw, cbuf.before)
