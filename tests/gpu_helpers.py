"""Helpers for the GPU parity tests: device buffers with guard bands, calls
through the C ABI, and comparison against the CPU oracle."""

from __future__ import annotations

import contextlib
import functools

import numpy as np

import bm_inputs as gen
import oracle

F32_CANARY = np.uint32(0x7FFADBAD)   # a quiet-NaN payload that no computation produces
BF16_CANARY = np.uint16(0x7FBD)


def torch():
    import torch as _t
    return _t


def bf16_to_device(bits: np.ndarray):
    t = torch()
    return t.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(t.bfloat16).cuda()


def u8_to_device(codes: np.ndarray):
    t = torch()
    return t.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8)).cuda()


def f32_to_device(x: np.ndarray):
    t = torch()
    return t.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).cuda()


def device_to_numpy(x):
    t = torch()
    if x.dtype == t.bfloat16:
        return x.view(t.int16).cpu().numpy().view(np.uint16)
    return x.cpu().numpy()


@functools.lru_cache(maxsize=32)
def cached_bf16(rows, cols, dist, seed, std=1.0, lo=-1.0, hi=1.0):
    out = gen.matrix_bf16(rows, cols, dist, seed, std, lo, hi)
    out.setflags(write=False)
    return out


def operand(rows, cols, dist="normal", seed=1, std=1.0, lo=-1.0, hi=1.0, pad=0):
    """bf16 bits [rows, cols + pad]; the padding holds NaN (it must never be read)."""
    bits = cached_bf16(rows, cols, dist, seed, std, lo, hi)
    if pad:
        return gen.pad_ld(bits, cols + pad, gen.BF16_NAN)
    return np.array(bits)


class CBuffer:
    """An output C of m x n inside an (m + extra_rows) x ldc buffer of canaries."""

    def __init__(self, m, n, ldc, bf16, init=None, extra_rows=2):
        self.m, self.n, self.ldc, self.bf16 = m, n, ldc, bf16
        rows = m + extra_rows
        if bf16:
            host = np.full((rows, ldc), BF16_CANARY, np.uint16)
        else:
            host = np.full((rows, ldc), F32_CANARY, np.uint32).view(np.float32)
        if init is not None:
            host[:m, :n] = init
        self.before = host.copy()
        self.dev = bf16_to_device(host) if bf16 else f32_to_device(host)

    @property
    def ptr(self):
        return self.dev.data_ptr()

    def result(self):
        """(values as float64 [m, n], full raw buffer)."""
        raw = device_to_numpy(self.dev)
        vals = raw[:self.m, :self.n]
        vals = gen.bf16_bits_to_f32(vals).astype(np.float64) if self.bf16 else vals.astype(np.float64)
        return vals, raw

    def raw_bits(self, raw):
        return raw if self.bf16 else raw.view(np.uint32)

    def assert_guard_intact(self, raw, mask_written=None):
        """Everything outside [m, n] (and outside mask_written inside it) is bit-identical."""
        before = self.raw_bits(self.before)
        after = self.raw_bits(raw)
        outside = np.ones(after.shape, bool)
        outside[:self.m, :self.n] = False
        if mask_written is not None:
            outside[:self.m, :self.n] = ~mask_written
        bad = np.argwhere(outside & (before != after))
        assert bad.size == 0, f"{len(bad)} elements outside the output changed, first at {bad[0]}"


def c_input_values(c_init, bf16):
    if c_init is None:
        return None
    return gen.bf16_bits_to_f32(c_init).astype(np.float64) if bf16 else np.asarray(c_init, np.float64)


def check_no_device_error():
    import blas3_tensor_core_gb300 as bm
    st = bm.bm_get_last_device_error(torch().cuda.current_stream().cuda_stream)
    assert st == bm.BM_OK, bm.bm_status_string(st)


def run_gemm(m, n, k, ta, tb, alpha, A, B, beta, cbuf: CBuffer, workspace=None):
    import blas3_tensor_core_gb300 as bm
    t = torch()
    dA = bf16_to_device(A)
    dB = bf16_to_device(B)
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        ws_ptr, ws_bytes = workspace.data_ptr(), workspace.numel() * workspace.element_size()
    st = bm.bm_gemm_bf16(m, n, k, ta, tb, alpha, dA.data_ptr(), A.shape[1], dB.data_ptr(), B.shape[1],
                         beta, cbuf.ptr, cbuf.ldc, bm.BM_C_BF16 if cbuf.bf16 else bm.BM_C_F32,
                         ws_ptr, ws_bytes, t.cuda.current_stream().cuda_stream)
    assert st == bm.BM_OK, bm.bm_status_string(st)
    t.cuda.synchronize()
    check_no_device_error()
    return cbuf.result()


def _ws_args(workspace):
    if workspace is None:
        return None, 0
    return workspace.data_ptr(), workspace.numel() * workspace.element_size()


def run_syrk(uplo, trans, n, k, alpha, A, beta, cbuf: CBuffer, workspace=None):
    import blas3_tensor_core_gb300 as bm
    t = torch()
    dA = bf16_to_device(A)
    st = bm.bm_syrk_bf16(uplo, trans, n, k, alpha, dA.data_ptr(), A.shape[1], beta, cbuf.ptr, cbuf.ldc,
                         bm.BM_C_BF16 if cbuf.bf16 else bm.BM_C_F32, *_ws_args(workspace),
                         t.cuda.current_stream().cuda_stream)
    assert st == bm.BM_OK, bm.bm_status_string(st)
    t.cuda.synchronize()
    check_no_device_error()
    return cbuf.result()


def run_gemm_e4m3(m, n, k, alpha, A, B, beta, cbuf: CBuffer, workspace=None):
    """C = alpha * A B^T + beta * C with E4M3 codes A [m, k], B [n, k] (row lengths = leading dimensions)."""
    import blas3_tensor_core_gb300 as bm
    t = torch()
    dA = u8_to_device(A)
    dB = u8_to_device(B)
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        ws_ptr, ws_bytes = workspace.data_ptr(), workspace.numel() * workspace.element_size()
    st = bm.bm_gemm_e4m3(m, n, k, alpha, dA.data_ptr(), A.shape[1], dB.data_ptr(), B.shape[1], beta, cbuf.ptr,
                         cbuf.ldc, bm.BM_C_BF16 if cbuf.bf16 else bm.BM_C_F32, ws_ptr, ws_bytes,
                         t.cuda.current_stream().cuda_stream)
    assert st == bm.BM_OK, bm.bm_status_string(st)
    t.cuda.synchronize()
    check_no_device_error()
    return cbuf.result()


def mxfp8_tiled_scales(S, rows, k, pad_code=0):
    """UE8M0 codes S [rows, >= ceil(k/32)] (row-major) in the tiled atom layout the library reads;
    padding entries (rows past `rows`, groups past ceil(k/32)) hold pad_code."""
    import blas3_tensor_core_gb300 as bm
    groups = (k + 31) // 32
    out = np.full(bm.mxfp8_scale_bytes(rows, k), pad_code, np.uint8)
    r = np.repeat(np.arange(rows, dtype=np.int64), groups)
    g = np.tile(np.arange(groups, dtype=np.int64), rows)
    out[bm.mxfp8_scale_offset(r, g, k)] = np.asarray(S)[:rows, :groups].reshape(-1)
    return out


def run_gemm_mxfp8(m, n, k, alpha, A, SA, B, SB, beta, cbuf: CBuffer, workspace=None, pad_code=0):
    """C = alpha * (A . SA)(B . SB)^T + beta * C; A [m, k], B [n, k] E4M3 codes (row lengths = leading
    dimensions), SA [m, groups], SB [n, groups] UE8M0 codes, passed in the tiled layout."""
    import blas3_tensor_core_gb300 as bm
    t = torch()
    dA, dB = u8_to_device(A), u8_to_device(B)
    dSA = u8_to_device(mxfp8_tiled_scales(SA, m, k, pad_code))
    dSB = u8_to_device(mxfp8_tiled_scales(SB, n, k, pad_code))
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        ws_ptr, ws_bytes = workspace.data_ptr(), workspace.numel() * workspace.element_size()
    st = bm.bm_gemm_mxfp8(m, n, k, alpha, dA.data_ptr(), A.shape[1], dSA.data_ptr(), dB.data_ptr(), B.shape[1],
                          dSB.data_ptr(), beta, cbuf.ptr, cbuf.ldc, bm.BM_C_BF16 if cbuf.bf16 else bm.BM_C_F32,
                          ws_ptr, ws_bytes, t.cuda.current_stream().cuda_stream)
    assert st == bm.BM_OK, bm.bm_status_string(st)
    t.cuda.synchronize()
    check_no_device_error()
    return cbuf.result()


def run_syr2k(uplo, trans, n, k, alpha, A, B, beta, cbuf: CBuffer, workspace=None):
    import blas3_tensor_core_gb300 as bm
    t = torch()
    dA = bf16_to_device(A)
    dB = bf16_to_device(B)
    st = bm.bm_syr2k_bf16(uplo, trans, n, k, alpha, dA.data_ptr(), A.shape[1], dB.data_ptr(), B.shape[1], beta,
                          cbuf.ptr, cbuf.ldc, bm.BM_C_BF16 if cbuf.bf16 else bm.BM_C_F32, *_ws_args(workspace),
                          t.cuda.current_stream().cuda_stream)
    assert st == bm.BM_OK, bm.bm_status_string(st)
    t.cuda.synchronize()
    check_no_device_error()
    return cbuf.result()


def assert_parity(got, ref, bound, alpha, beta, c_in, out_bf16, what=""):
    ok, worst, where = oracle.compare(got, ref, bound, alpha, beta, c_in, out_bf16)
    if not ok:
        idx = tuple(int(x) for x in where)
        raise AssertionError(f"{what}: worst |err|/tol = {worst:.3g} at {idx}: "
                             f"got {np.asarray(got)[idx]!r} ref {np.asarray(ref)[idx]!r}")
    return worst


def tile_samples(m, n, tile_m=128, tile_n=256, per_tile=4, seed=0, extra=None):
    """Random positions: `per_tile` inside every output tile, plus the matrix corners."""
    rng = np.random.default_rng(seed)
    rows, cols = [], []
    for tm in range(0, m, tile_m):
        for tn in range(0, n, tile_n):
            h, w = min(tile_m, m - tm), min(tile_n, n - tn)
            rows.append(tm + rng.integers(0, h, per_tile))
            cols.append(tn + rng.integers(0, w, per_tile))
    corners_r = np.array([0, 0, m - 1, m - 1])
    corners_c = np.array([0, n - 1, 0, n - 1])
    rows.append(corners_r)
    cols.append(corners_c)
    if extra is not None:
        rows.append(extra[0])
        cols.append(extra[1])
    return np.concatenate(rows).astype(np.int64), np.concatenate(cols).astype(np.int64)


VARIANTS = [0, 1, 2, 3]          # automatic, 128x256 single SM, 128x128 single SM, 256x256 SM pair
VARIANT_IDS = ["auto", "single128x256", "single128x128", "pair256x256"]


@contextlib.contextmanager
def tile_variant(v):
    """Force one kernel variant for the calls inside the block (0 = automatic)."""
    import blas3_tensor_core_gb300 as bm
    assert bm.bm_set_tile_override(v) == bm.BM_OK
    try:
        yield
    finally:
        bm.bm_set_tile_override(0)
