"""Bounded waits: a stage whose copy is never issued makes the MMA warp's wait run
out. The kernel must record BM_ERR_TIMEOUT, free its tensor memory and exit, and
the CUDA context must stay usable for the next call. Nothing here faults or hangs
the GPU: the stall is a copy that is not issued, and every wait has a 50 ms limit.
"""

import numpy as np
import pytest

import oracle
from gpu_helpers import CBuffer, assert_parity, operand, tile_variant, torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from blas3_tensor_core_gb300 import build
    build.build()
    assert torch().cuda.is_available()


@pytest.mark.parametrize("beta", [0.0, 1.0], ids=["beta0", "beta1"])
@pytest.mark.parametrize("variant", [1, 3], ids=["single128x256", "pair256x256"])
def test_stalled_stage_reports_timeout_and_context_survives(variant, beta):
    """beta = 1 runs the epilogue halves that meet at named barriers: they leave together."""
    import blas3_tensor_core_gb300 as bm
    from gpu_helpers import bf16_to_device
    t = torch()
    m, n, k = 512, 512, 256
    A = operand(m, k, "normal", 1)
    B = operand(k, n, "normal", 2)
    dA, dB = bf16_to_device(A), bf16_to_device(B)
    stream = t.cuda.current_stream().cuda_stream
    cbuf = CBuffer(m, n, n, False, init=np.zeros((m, n), np.float32))
    assert bm.bm_get_last_device_error(stream) == bm.BM_OK
    bm.bm_set_wait_timeout_ms(50)
    bm.bm_debug_inject_stall(1)
    try:
        with tile_variant(variant):
            st = bm.bm_gemm_bf16(m, n, k, 0, 0, 1.0, dA.data_ptr(), k, dB.data_ptr(), n, beta, cbuf.ptr, n,
                                 bm.BM_C_F32, None, 0, stream)
            assert st == bm.BM_OK
            assert bm.bm_get_last_device_error(stream) == bm.BM_ERR_TIMEOUT
    finally:
        bm.bm_debug_inject_stall(0)
        bm.bm_set_wait_timeout_ms(2000)
    assert bm.bm_get_last_device_error(stream) == bm.BM_OK  # the word was cleared
    # the context and the tensor memory are still usable
    c0 = np.full((m, n), 0.5, np.float32)
    cbuf2 = CBuffer(m, n, n, False, init=c0)
    with tile_variant(variant):
        st = bm.bm_gemm_bf16(m, n, k, 0, 0, 1.0, dA.data_ptr(), k, dB.data_ptr(), n, beta, cbuf2.ptr, n,
                             bm.BM_C_F32, None, 0, stream)
    assert st == bm.BM_OK
    assert bm.bm_get_last_device_error(stream) == bm.BM_OK
    got, raw = cbuf2.result()
    rows = np.arange(0, m, 7)
    cols = (rows * 13) % n
    ref, bound = oracle.default().gemm_entries(k, 0, 0, 1.0, A, B, rows, cols, beta, c0)
    c_in = c0[rows, cols].astype(np.float64) if beta != 0 else None
    assert_parity(got[rows, cols], ref, bound, 1.0, beta, c_in, False, "after timeout")
    cbuf2.assert_guard_intact(raw)
