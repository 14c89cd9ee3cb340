"""The GEMM entry point that allocates nothing, bm_gemm_bf16_noalloc, on a GB300.

Some callers cannot call cudaMalloc: a framework that owns all device memory
through its own pool, a plug-in called back by another library without an
allocator, or a latency-critical path that cannot afford cudaMalloc's implicit
synchronisation. For them the library keeps its split-K scratch in a static
device array. These tests call that entry point through the C ABI and compare
it with bm_gemm_bf16 given a caller-owned workspace, and with the CPU oracle,
on two calls in a row (the array keeps the previous call's contents). A shape
whose full split would not fit the array is split fewer ways, exactly as
bm_gemm_bf16 splits it with a workspace of the array's size. A call that is the
first use of the library in a process, so that no device status word exists
yet, still returns cleanly from a device-side wait that runs out.

The file name sorts last so that a run that stops at the first failure has
already run every other test. It depends on no state left by other tests.
"""

import os
import subprocess
import sys
import textwrap

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


def _oracle_check(got, m, n, k, A, B, alpha, beta, c_init, bf16, what):
    ref, bound = oracle.default().gemm(m, n, k, 0, 0, alpha, A, B, beta, c_init if beta != 0 else None)
    c_in = None
    if beta != 0:
        c_in = gen.bf16_bits_to_f32(c_init).astype(np.float64) if bf16 else np.asarray(c_init, np.float64)
    ok, worst, where = oracle.compare(got, ref, bound, alpha, beta, c_in, bf16)
    assert ok, (what, worst, where)


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
        _oracle_check(got, m, n, k, A, B, 1.0, 0.0, None, True, f"seed {seed}")


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


@pytest.mark.parametrize("beta", [0.0, -1.0])
def test_n_half_tail_without_allocation_exact(beta):
    """2560 x 2048 x 1024: the 4 tail tiles run as N halves (no partials), which needs no
    scratch at all; the allocation-free call matches the oracle on every element and the
    workspace entry point bit for bit."""
    import blas3_tensor_core_gb300 as bm
    m, n, k = 2560, 2048, 1024
    st, plan = bm.bm_gemm_bf16_plan(m, n, k, bm.bm_gemm_bf16_workspace_size(m, n, k))
    assert (plan.split_tiles, plan.k_splits, plan.n_splits, plan.workspace_bytes) == (4, 1, 2, 0)
    A = operand(m, k, "int", 97, lo=-3, hi=3)
    B = operand(k, n, "int", 98, lo=-3, hi=3)
    c0 = gen.integers(99, m * n, -30, 30).reshape(m, n).astype(np.float32)
    dA, dB = bf16_to_device(A), bf16_to_device(B)
    want, _ = _with_workspace(m, n, k, dA, dB, k, n, 1.0, beta, c0, False)
    got = _noalloc(m, n, k, dA, dB, k, n, 1.0, beta, c0, False)
    assert np.array_equal(got, want)
    _oracle_check(got, m, n, k, A, B, 1.0, beta, c0, False, f"beta {beta}")


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
        _oracle_check(got, m, n, k, A, B, -0.5, 1.5, c0, False, "beta 1.5")


def test_full_split_beyond_the_array_splits_fewer_ways():
    """512 x 1024 x 8192: a 10-way split of the 16 tiles would need 21.0 MB of partials; within
    the 16 MiB array the planner splits 8 ways, as bm_gemm_bf16 does with a 16 MiB workspace.
    Both entry points then run the same plan, so they agree bit for bit, twice in a row."""
    import blas3_tensor_core_gb300 as bm
    t = torch()
    m, n, k = 512, 1024, 8192
    assert bm.bm_gemm_bf16_workspace_size(m, n, k) > bm.BM_NOALLOC_SCRATCH_BYTES
    plan = bm.bm_gemm_bf16_plan(m, n, k, bm.BM_NOALLOC_SCRATCH_BYTES)[1]
    assert plan.k_splits > 1 and plan.workspace_bytes <= bm.BM_NOALLOC_SCRATCH_BYTES
    ws = t.empty(bm.BM_NOALLOC_SCRATCH_BYTES // 4, dtype=t.float32, device="cuda")
    for seed in (41, 51):
        A = operand(m, k, "normal", seed)
        B = operand(k, n, "normal", seed + 1)
        dA, dB = bf16_to_device(A), bf16_to_device(B)
        cw = CBuffer(m, n, n, True, init=np.zeros((m, n), np.uint16))
        st = bm.bm_gemm_bf16(m, n, k, 0, 0, 1.0, dA.data_ptr(), k, dB.data_ptr(), n, 0.0, cw.ptr, n,
                             bm.BM_C_BF16, ws.data_ptr(), bm.BM_NOALLOC_SCRATCH_BYTES,
                             t.cuda.current_stream().cuda_stream)
        assert st == bm.BM_OK
        t.cuda.synchronize()
        want = cw.result()[0]
        got = _noalloc(m, n, k, dA, dB, k, n, 1.0, 0.0, None, True)
        assert np.array_equal(got, want), seed
        _oracle_check(got, m, n, k, A, B, 1.0, 0.0, None, True, f"seed {seed}")


_FRESH_PROCESS = textwrap.dedent("""
    import sys
    import numpy as np
    import torch
    sys.path.insert(0, {root!r})
    sys.path.insert(0, {tests!r})
    import blas3_tensor_core_gb300 as bm
    import oracle
    from gpu_helpers import CBuffer, bf16_to_device, operand
    torch.cuda.set_device(0)
    h = torch.cuda.current_stream().cuda_stream
    m, n, k = 512, 512, 256
    A = operand(m, k, "normal", 1)
    B = operand(k, n, "normal", 2)
    dA, dB = bf16_to_device(A), bf16_to_device(B)
    c = CBuffer(m, n, n, False, init=np.zeros((m, n), np.float32))
    bm.bm_set_wait_timeout_ms(50)
    bm.bm_debug_inject_stall(1)
    # the first call of the library in this process: no status word exists on the device
    st = bm.bm_gemm_bf16_noalloc(m, n, k, 0, 0, 1.0, dA.data_ptr(), k, dB.data_ptr(), n, 0.0, c.ptr, n,
                                 bm.BM_C_F32, h)
    assert st == bm.BM_OK, st
    torch.cuda.synchronize()   # the stalled kernel gave up and exited; nothing faulted
    bm.bm_debug_inject_stall(0)
    bm.bm_set_wait_timeout_ms(2000)
    # the timeout had no status word to go to: the word created now starts clear
    assert bm.bm_get_last_device_error(h) == bm.BM_OK
    for entry in ("noalloc", "workspace"):
        c2 = CBuffer(m, n, n, False, init=np.zeros((m, n), np.float32))
        if entry == "noalloc":
            st = bm.bm_gemm_bf16_noalloc(m, n, k, 0, 0, 1.0, dA.data_ptr(), k, dB.data_ptr(), n, 0.0, c2.ptr,
                                         n, bm.BM_C_F32, h)
        else:
            st = bm.bm_gemm_bf16(m, n, k, 0, 0, 1.0, dA.data_ptr(), k, dB.data_ptr(), n, 0.0, c2.ptr, n,
                                 bm.BM_C_F32, None, 0, h)
        assert st == bm.BM_OK, st
        assert bm.bm_get_last_device_error(h) == bm.BM_OK
        got, raw = c2.result()
        ref, bound = oracle.default().gemm(m, n, k, 0, 0, 1.0, A, B)
        ok, worst, _ = oracle.compare(got, ref, bound, 1.0)
        assert ok, (entry, worst)
        c2.assert_guard_intact(raw)
    print("fresh-process noalloc timeout ok")
""")


def test_first_call_without_status_word_survives_a_wait_limit():
    """A device-side wait that runs out in a call made before any status word exists on
    the device (the allocation-free entry point never creates one): the kernel gives
    up after its 50 ms limit, frees its tensor memory and exits; the call's timeout is
    recorded nowhere, and the context stays usable for both entry points. Run in a
    fresh process so that no earlier test has created the word. The stall is a copy
    that is never issued; nothing faults or hangs."""
    tests = os.path.dirname(os.path.abspath(__file__))
    root = os.path.dirname(tests)
    script = _FRESH_PROCESS.format(root=root, tests=tests)
    res = subprocess.run([sys.executable, "-c", script], capture_output=True, text=True, timeout=600)
    assert res.returncode == 0, res.stdout[-2000:] + res.stderr[-4000:]
    assert "fresh-process noalloc timeout ok" in res.stdout
