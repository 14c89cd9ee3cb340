"""GB300 (sm_103a) BF16 GEMM / SYRK: Python binding of the C ABI in include/bm.h.

The functions named ``bm_*`` mirror the C entry points one to one (plain
integers for pointers and the stream). ``gemm`` and ``syrk`` are conveniences
that read sizes, leading dimensions and the current stream from torch tensors
and call the same entry points. Nothing here computes: every step of the path
runs in the CUDA library, and a missing library raises instead of falling
back.
"""

from __future__ import annotations

import ctypes
import os
import threading

__all__ = [
    "BMError", "library", "library_path",
    "BM_OK", "BM_ERR_INVALID_VALUE", "BM_ERR_MISALIGNED", "BM_ERR_ARCH", "BM_ERR_CUDA",
    "BM_ERR_TIMEOUT", "BM_ERR_WORKSPACE", "BM_OP_N", "BM_OP_T", "BM_C_F32", "BM_C_BF16",
    "BM_LOWER", "BM_UPPER", "Plan",
    "bm_gemm_bf16", "bm_gemm_bf16_noalloc", "BM_NOALLOC_SCRATCH_BYTES", "bm_syrk_bf16", "bm_syr2k_bf16",
    "bm_gemm_e4m3", "bm_gemm_e4m3_workspace_size", "bm_gemm_mxfp8", "bm_gemm_mxfp8_workspace_size",
    "bm_gemm_mxfp8_plan", "bm_quantize_mxfp8", "mxfp8_scale_bytes", "mxfp8_scale_offset", "bm_gemm_bf16_workspace_size", "bm_get_last_device_error",
    "bm_set_wait_timeout_ms", "bm_debug_inject_stall", "bm_status_string", "bm_gemm_bf16_plan",
    "bm_syrk_bf16_plan", "bm_syrk_bf16_tile_order", "bm_syrk_bf16_workspace_size",
    "bm_syr2k_bf16_workspace_size", "bm_set_tile_override", "bm_version", "gemm", "syrk", "syr2k", "workspace_size",
]

BM_OK, BM_ERR_INVALID_VALUE, BM_ERR_MISALIGNED, BM_ERR_ARCH, BM_ERR_CUDA, BM_ERR_TIMEOUT, BM_ERR_WORKSPACE = range(7)
BM_OP_N, BM_OP_T = 0, 1
BM_C_F32, BM_C_BF16 = 0, 1
BM_LOWER, BM_UPPER = 0, 1

_HERE = os.path.dirname(os.path.abspath(__file__))
library_path = os.path.join(_HERE, "libbm.so")
_lib = None
_lock = threading.Lock()

_i64, _i32, _u32, _f32, _vp, _sz = (ctypes.c_int64, ctypes.c_int, ctypes.c_uint32, ctypes.c_float,
                                    ctypes.c_void_p, ctypes.c_size_t)


class Plan(ctypes.Structure):
    _fields_ = [("tile_m", ctypes.c_int32), ("tile_n", ctypes.c_int32), ("tile_k", ctypes.c_int32),
                ("stages", ctypes.c_int32), ("tiles", ctypes.c_int64), ("k_splits", ctypes.c_int32),
                ("ctas", ctypes.c_int32), ("cta_pair", ctypes.c_int32), ("kernels", ctypes.c_int32),
                ("workspace_bytes", ctypes.c_size_t), ("split_tiles", ctypes.c_int64),
                ("stage_kblocks", ctypes.c_int32), ("n_splits", ctypes.c_int32)]

    def as_dict(self):
        return {f: getattr(self, f) for f, _ in self._fields_}


class BMError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {bm_status_string(status)} ({status})")


def library():
    """The loaded CUDA library; raises if it has not been built."""
    global _lib
    if _lib is None:
        with _lock:
            if _lib is None:
                if not os.path.exists(library_path):
                    raise RuntimeError(
                        f"CUDA library not built: {library_path} is missing "
                        "(run `python -m blas3_tensor_core_gb300.build`)")
                lib = ctypes.CDLL(library_path)
                lib.bm_gemm_bf16.argtypes = [_i64, _i64, _i64, _i32, _i32, _f32, _vp, _i64, _vp, _i64,
                                             _f32, _vp, _i64, _i32, _vp, _sz, _vp]
                lib.bm_gemm_bf16.restype = _i32
                lib.bm_gemm_bf16_noalloc.argtypes = [_i64, _i64, _i64, _i32, _i32, _f32, _vp, _i64, _vp, _i64,
                                                     _f32, _vp, _i64, _i32, _vp]
                lib.bm_gemm_bf16_noalloc.restype = _i32
                lib.bm_gemm_e4m3.argtypes = [_i64, _i64, _i64, _f32, _vp, _i64, _vp, _i64, _f32, _vp, _i64, _i32,
                                             _vp, _sz, _vp]
                lib.bm_gemm_e4m3.restype = _i32
                lib.bm_gemm_e4m3_workspace_size.argtypes = [_i64, _i64, _i64]
                lib.bm_gemm_e4m3_workspace_size.restype = _sz
                lib.bm_gemm_mxfp8.argtypes = [_i64, _i64, _i64, _f32, _vp, _i64, _vp, _vp, _i64, _vp, _f32, _vp,
                                              _i64, _i32, _vp, _sz, _vp]
                lib.bm_gemm_mxfp8.restype = _i32
                lib.bm_gemm_mxfp8_workspace_size.argtypes = [_i64, _i64, _i64]
                lib.bm_gemm_mxfp8_workspace_size.restype = _sz
                lib.bm_gemm_mxfp8_plan.argtypes = [_i64, _i64, _i64, _sz, ctypes.POINTER(Plan)]
                lib.bm_gemm_mxfp8_plan.restype = _i32
                lib.bm_quantize_mxfp8.argtypes = [_i64, _i64, _vp, _i64, _vp, _i64, _vp, _vp]
                lib.bm_quantize_mxfp8.restype = _i32
                lib.bm_syrk_bf16.argtypes = [_i32, _i32, _i64, _i64, _f32, _vp, _i64, _f32, _vp, _i64,
                                             _i32, _vp, _sz, _vp]
                lib.bm_syrk_bf16.restype = _i32
                lib.bm_syr2k_bf16.argtypes = [_i32, _i32, _i64, _i64, _f32, _vp, _i64, _vp, _i64, _f32, _vp,
                                              _i64, _i32, _vp, _sz, _vp]
                lib.bm_syr2k_bf16.restype = _i32
                lib.bm_syrk_bf16_workspace_size.argtypes = [_i32, _i64, _i64]
                lib.bm_syrk_bf16_workspace_size.restype = _sz
                lib.bm_syr2k_bf16_workspace_size.argtypes = [_i32, _i64, _i64]
                lib.bm_syr2k_bf16_workspace_size.restype = _sz
                lib.bm_gemm_bf16_workspace_size.argtypes = [_i64, _i64, _i64]
                lib.bm_gemm_bf16_workspace_size.restype = _sz
                lib.bm_get_last_device_error.argtypes = [_vp]
                lib.bm_get_last_device_error.restype = _i32
                lib.bm_set_wait_timeout_ms.argtypes = [_u32]
                lib.bm_set_wait_timeout_ms.restype = None
                lib.bm_debug_inject_stall.argtypes = [_i32]
                lib.bm_debug_inject_stall.restype = None
                lib.bm_status_string.argtypes = [_i32]
                lib.bm_status_string.restype = ctypes.c_char_p
                lib.bm_gemm_bf16_plan.argtypes = [_i64, _i64, _i64, _sz, ctypes.POINTER(Plan)]
                lib.bm_gemm_bf16_plan.restype = _i32
                lib.bm_syrk_bf16_plan.argtypes = [_i32, _i64, _i64, _sz, ctypes.POINTER(Plan)]
                lib.bm_syrk_bf16_plan.restype = _i32
                lib.bm_syrk_bf16_tile_order.argtypes = [_i32, _i64, _i64, _i64, _vp, _vp]
                lib.bm_syrk_bf16_tile_order.restype = _i32
                lib.bm_set_tile_override.argtypes = [_i32]
                lib.bm_set_tile_override.restype = _i32
                lib.bm_version.argtypes = []
                lib.bm_version.restype = _i32
                _lib = lib
    return _lib


# -- the C ABI, name for name -------------------------------------------------------
def bm_gemm_bf16(m, n, k, transA, transB, alpha, A, lda, B, ldb, beta, C, ldc, c_type,
                 workspace=None, workspace_bytes=0, stream=None) -> int:
    return library().bm_gemm_bf16(m, n, k, transA, transB, alpha, A, lda, B, ldb, beta, C, ldc,
                                  c_type, workspace, workspace_bytes, stream)


# Size of the device array that bm_gemm_bf16_noalloc uses for split-K partials.
BM_NOALLOC_SCRATCH_BYTES = 16 * 1024 * 1024


def bm_gemm_bf16_noalloc(m, n, k, transA, transB, alpha, A, lda, B, ldb, beta, C, ldc, c_type,
                         stream=None) -> int:
    """The GEMM entry point that allocates nothing (split-K scratch is a static device array)."""
    return library().bm_gemm_bf16_noalloc(m, n, k, transA, transB, alpha, A, lda, B, ldb, beta, C, ldc,
                                          c_type, stream)


def bm_syrk_bf16(uplo, trans, n, k, alpha, A, lda, beta, C, ldc, c_type, workspace=None, workspace_bytes=0,
                 stream=None) -> int:
    return library().bm_syrk_bf16(uplo, trans, n, k, alpha, A, lda, beta, C, ldc, c_type, workspace,
                                  workspace_bytes, stream)


def bm_syrk_bf16_workspace_size(uplo, n, k) -> int:
    return library().bm_syrk_bf16_workspace_size(uplo, n, k)


def bm_syr2k_bf16_workspace_size(uplo, n, k) -> int:
    return library().bm_syr2k_bf16_workspace_size(uplo, n, k)


def bm_gemm_e4m3(m, n, k, alpha, A, lda, B, ldb, beta, C, ldc, c_type, workspace=None, workspace_bytes=0,
                 stream=None) -> int:
    return library().bm_gemm_e4m3(m, n, k, alpha, A, lda, B, ldb, beta, C, ldc, c_type, workspace,
                                  workspace_bytes, stream)


def bm_gemm_e4m3_workspace_size(m, n, k) -> int:
    return library().bm_gemm_e4m3_workspace_size(m, n, k)


def bm_gemm_mxfp8(m, n, k, alpha, A, lda, SA, B, ldb, SB, beta, C, ldc, c_type, workspace=None,
                  workspace_bytes=0, stream=None) -> int:
    return library().bm_gemm_mxfp8(m, n, k, alpha, A, lda, SA, B, ldb, SB, beta, C, ldc, c_type, workspace,
                                   workspace_bytes, stream)


def bm_gemm_mxfp8_workspace_size(m, n, k) -> int:
    return library().bm_gemm_mxfp8_workspace_size(m, n, k)


def bm_gemm_mxfp8_plan(m, n, k, workspace_bytes=0):
    plan = Plan()
    st = library().bm_gemm_mxfp8_plan(m, n, k, workspace_bytes, ctypes.byref(plan))
    return st, plan


def bm_quantize_mxfp8(rows, k, X, ldx, Q, ldq, S, stream=None) -> int:
    return library().bm_quantize_mxfp8(rows, k, X, ldx, Q, ldq, S, stream)


def mxfp8_scale_bytes(rows, k) -> int:
    """Size of an MXFP8 scale array in the tiled layout: ceil(rows/128) x ceil(k/128) atoms of 512 bytes."""
    return -(-rows // 128) * -(-k // 128) * 512


def mxfp8_scale_offset(r, g, k):
    """Byte offset of the scale of row r, group g (elements 32 g .. 32 g + 31) in the tiled layout
    (works elementwise on NumPy integer arrays)."""
    katoms = -(-k // 128)
    return ((r // 128) * katoms + g // 4) * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + g % 4


def bm_syr2k_bf16(uplo, trans, n, k, alpha, A, lda, B, ldb, beta, C, ldc, c_type, workspace=None,
                  workspace_bytes=0, stream=None) -> int:
    return library().bm_syr2k_bf16(uplo, trans, n, k, alpha, A, lda, B, ldb, beta, C, ldc, c_type, workspace,
                                   workspace_bytes, stream)


def bm_gemm_bf16_workspace_size(m, n, k) -> int:
    return library().bm_gemm_bf16_workspace_size(m, n, k)


def bm_get_last_device_error(stream=None) -> int:
    return library().bm_get_last_device_error(stream)


def bm_set_wait_timeout_ms(ms: int) -> None:
    library().bm_set_wait_timeout_ms(ms)


def bm_debug_inject_stall(enable: int) -> None:
    library().bm_debug_inject_stall(1 if enable else 0)


def bm_status_string(status: int) -> str:
    return library().bm_status_string(status).decode()


def bm_gemm_bf16_plan(m, n, k, workspace_bytes=0):
    plan = Plan()
    st = library().bm_gemm_bf16_plan(m, n, k, workspace_bytes, ctypes.byref(plan))
    return st, plan


def bm_syrk_bf16_plan(uplo, n, k, workspace_bytes=0):
    plan = Plan()
    st = library().bm_syrk_bf16_plan(uplo, n, k, workspace_bytes, ctypes.byref(plan))
    return st, plan


def bm_syrk_bf16_tile_order(uplo, n, k):
    """(status, tile rows, tile columns) of the SYRK schedule, as int64 NumPy arrays."""
    import numpy as np
    st, plan = bm_syrk_bf16_plan(uplo, n, k)
    rows = np.zeros(max(plan.tiles, 0), np.int64)
    cols = np.zeros(max(plan.tiles, 0), np.int64)
    if st != BM_OK:
        return st, rows, cols
    st = library().bm_syrk_bf16_tile_order(uplo, n, k, plan.tiles, rows.ctypes.data, cols.ctypes.data)
    return st, rows, cols


TILE_AUTO, TILE_SINGLE_128x256, TILE_SINGLE_128x128, TILE_PAIR_256x256 = range(4)


def bm_set_tile_override(variant: int) -> int:
    return library().bm_set_tile_override(variant)


def bm_version() -> int:
    return library().bm_version()


# -- torch conveniences (argument marshalling only) ------------------------------------
def _check(status: int, where: str) -> None:
    if status != BM_OK:
        raise BMError(status, where)


def _rowmajor_ld(t, name):
    if t.dim() != 2 or t.stride(1) != 1:
        raise ValueError(f"{name} must be a 2-D row-major tensor (unit column stride)")
    return max(t.stride(0), 1)


def _on_current_device(**tensors):
    """Every tensor must live on the current CUDA device: the library launches there and takes
    the pointers as device addresses."""
    import torch
    for name, t in tensors.items():
        if t is None:
            continue
        if not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor (got device {t.device})")
    current = torch.cuda.current_device()
    for name, t in tensors.items():
        if t is not None and t.device.index != current:
            raise ValueError(f"{name} is on {t.device}, the current device is cuda:{current}")


def _stream_handle(stream):
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def _ctype(C):
    import torch
    if C.dtype == torch.float32:
        return BM_C_F32
    if C.dtype == torch.bfloat16:
        return BM_C_BF16
    raise TypeError("C must be float32 or bfloat16")


def workspace_size(m, n, k) -> int:
    return bm_gemm_bf16_workspace_size(m, n, k)


def gemm(A, B, C, alpha=1.0, beta=0.0, transA=False, transB=False, workspace=None, stream=None):
    """C = alpha * op(A) @ op(B) + beta * C on torch CUDA tensors (row-major, bf16 A/B)."""
    import torch
    if A.dtype != torch.bfloat16 or B.dtype != torch.bfloat16:
        raise TypeError("A and B must be bfloat16")
    m, n = C.shape
    k = A.shape[0] if transA else A.shape[1]
    if (A.shape[1] if transA else A.shape[0]) != m or (B.shape[1] if transB else B.shape[0]) != k \
            or (B.shape[0] if transB else B.shape[1]) != n:
        raise ValueError("inconsistent shapes")
    _on_current_device(A=A, B=B, C=C, workspace=workspace)
    ws_ptr, ws_bytes = (None, 0) if workspace is None else (workspace.data_ptr(),
                                                              workspace.numel() * workspace.element_size())
    st = bm_gemm_bf16(m, n, k, int(bool(transA)), int(bool(transB)), float(alpha),
                      A.data_ptr(), _rowmajor_ld(A, "A"), B.data_ptr(), _rowmajor_ld(B, "B"),
                      float(beta), C.data_ptr(), _rowmajor_ld(C, "C"), _ctype(C),
                      ws_ptr, ws_bytes, _stream_handle(stream))
    _check(st, "bm_gemm_bf16")
    return C


def _ws(workspace):
    if workspace is None:
        return None, 0
    return workspace.data_ptr(), workspace.numel() * workspace.element_size()


def syr2k(A, B, C, alpha=1.0, beta=0.0, uplo="L", trans=False, workspace=None, stream=None):
    """One triangle of C = alpha * (op(A) op(B)^T + op(B) op(A)^T) + beta * C (row-major, bf16 A, B)."""
    import torch
    if A.dtype != torch.bfloat16 or B.dtype != torch.bfloat16:
        raise TypeError("A and B must be bfloat16")
    if A.shape != B.shape:
        raise ValueError("A and B must have the same shape")
    n = C.shape[0]
    if C.shape[1] != n:
        raise ValueError("C must be square")
    k = A.shape[0] if trans else A.shape[1]
    if (A.shape[1] if trans else A.shape[0]) != n:
        raise ValueError("inconsistent shapes")
    lo = BM_LOWER if str(uplo).upper().startswith("L") else BM_UPPER
    _on_current_device(A=A, B=B, C=C, workspace=workspace)
    st = bm_syr2k_bf16(lo, int(bool(trans)), n, k, float(alpha), A.data_ptr(), _rowmajor_ld(A, "A"),
                       B.data_ptr(), _rowmajor_ld(B, "B"), float(beta), C.data_ptr(), _rowmajor_ld(C, "C"),
                       _ctype(C), *_ws(workspace), _stream_handle(stream))
    _check(st, "bm_syr2k_bf16")
    return C


def syrk(A, C, alpha=1.0, beta=0.0, uplo="L", trans=False, workspace=None, stream=None):
    """One triangle of C = alpha * op(A) @ op(A)^T + beta * C (row-major, bf16 A)."""
    import torch
    if A.dtype != torch.bfloat16:
        raise TypeError("A must be bfloat16")
    n = C.shape[0]
    if C.shape[1] != n:
        raise ValueError("C must be square")
    k = A.shape[0] if trans else A.shape[1]
    if (A.shape[1] if trans else A.shape[0]) != n:
        raise ValueError("inconsistent shapes")
    lo = BM_LOWER if str(uplo).upper().startswith("L") else BM_UPPER
    _on_current_device(A=A, C=C, workspace=workspace)
    st = bm_syrk_bf16(lo, int(bool(trans)), n, k, float(alpha), A.data_ptr(), _rowmajor_ld(A, "A"),
                      float(beta), C.data_ptr(), _rowmajor_ld(C, "C"), _ctype(C), *_ws(workspace),
                      _stream_handle(stream))
    _check(st, "bm_syrk_bf16")
    return C
