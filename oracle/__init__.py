"""CPU oracle for the BF16 GEMM / SYRK path (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and the bench's CPU-baseline leg use
this package. It wraps ``bm_oracle.c`` (plain double-precision triple loops,
compiled with gcc + OpenMP) through ctypes, and states the acceptance rule used
to compare the CUDA path against it.

Acceptance rule (per output element):

    |C - ref| <= 1e-3 * |alpha| * bound          (FP32 output)
               + 2^-8 * |ref|                     (BF16 output: one rounding)
               + 2^-20 * |beta * C_in|            (FP32 combine of beta * C)

``bound = sum_p |op(A)[i][p] * op(B)[p][j]|`` (for SYR2K the sum runs over both
products). The first term is the stated
tolerance for a k-term FP32 accumulation; the second is the unit roundoff of a
round-to-nearest-even cast to bfloat16; the third covers the few FP32
operations of the alpha/beta combine (unit roundoff 2^-24 each), which the
first term omits when alpha*bound is small next to beta*C.

Parity unpinned: none. Every function here is pinned by the tests in
``tests/test_oracle_pins.py`` (brute force in exact integer and rational
arithmetic, closed forms, NumPy float64 matmul, every E4M3 code, the OCP MX
conversion's ties, saturation and special groups, and the invariants A*I = A,
(A*B)^T = B^T*A^T, SYRK = one triangle of GEMM(A, A^T), SYR2K = one triangle of
GEMM(A, B^T) + GEMM(B, A^T), SYR2K(A, A) = 2 SYRK(A), beta-accumulation = sum of
two beta=0 calls).
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "bm_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libbm_oracle.so")

_lock = threading.Lock()
_default = None

_c_i64 = ctypes.c_int64
_c_int = ctypes.c_int
_c_dbl = ctypes.c_double
_c_vp = ctypes.c_void_p


def compile_oracle(src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile the C oracle into a shared object (gcc -O2 -fopenmp, portable flags)."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-Wall",
           src, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    os.replace(tmp, out)
    return out


def _needs_build(lib: str, src: str) -> bool:
    return (not os.path.exists(lib)) or os.path.getmtime(lib) < os.path.getmtime(src)


class Oracle:
    """ctypes handle on one compiled oracle library."""

    def __init__(self, lib_path: str):
        self.path = lib_path
        lib = ctypes.CDLL(lib_path)
        lib.oracle_num_threads.restype = _c_int
        lib.oracle_set_num_threads.argtypes = [_c_int]
        lib.oracle_gemm.argtypes = [_c_i64, _c_i64, _c_i64, _c_int, _c_int, _c_dbl,
                                    _c_vp, _c_i64, _c_vp, _c_i64, _c_dbl,
                                    _c_vp, _c_i64, _c_int, _c_vp, _c_vp, _c_i64]
        lib.oracle_gemm_entries.argtypes = [_c_i64, _c_int, _c_int, _c_dbl,
                                            _c_vp, _c_i64, _c_vp, _c_i64, _c_dbl,
                                            _c_vp, _c_i64, _c_int, _c_i64, _c_vp, _c_vp,
                                            _c_vp, _c_vp]
        lib.oracle_syrk.argtypes = [_c_int, _c_int, _c_i64, _c_i64, _c_dbl, _c_vp, _c_i64,
                                    _c_dbl, _c_vp, _c_i64, _c_int, _c_vp, _c_vp, _c_i64]
        lib.oracle_syrk_entries.argtypes = [_c_int, _c_int, _c_i64, _c_dbl, _c_vp, _c_i64,
                                            _c_dbl, _c_vp, _c_i64, _c_int, _c_i64, _c_vp,
                                            _c_vp, _c_vp, _c_vp]
        lib.oracle_syr2k.argtypes = [_c_int, _c_int, _c_i64, _c_i64, _c_dbl, _c_vp, _c_i64, _c_vp, _c_i64,
                                     _c_dbl, _c_vp, _c_i64, _c_int, _c_vp, _c_vp, _c_i64]
        lib.oracle_syr2k_entries.argtypes = [_c_int, _c_int, _c_i64, _c_dbl, _c_vp, _c_i64, _c_vp, _c_i64,
                                             _c_dbl, _c_vp, _c_i64, _c_int, _c_i64, _c_vp, _c_vp, _c_vp,
                                             _c_vp]
        lib.oracle_gemm_e4m3.argtypes = [_c_i64, _c_i64, _c_i64, _c_dbl, _c_vp, _c_i64, _c_vp, _c_i64,
                                         _c_dbl, _c_vp, _c_i64, _c_int, _c_vp, _c_vp, _c_i64]
        lib.oracle_gemm_e4m3_entries.argtypes = [_c_i64, _c_dbl, _c_vp, _c_i64, _c_vp, _c_i64, _c_dbl,
                                                 _c_vp, _c_i64, _c_int, _c_i64, _c_vp, _c_vp, _c_vp,
                                                 _c_vp]
        lib.oracle_gemm_mxfp8.argtypes = [_c_i64, _c_i64, _c_i64, _c_dbl, _c_vp, _c_i64, _c_vp, _c_i64,
                                          _c_vp, _c_i64, _c_vp, _c_i64, _c_dbl, _c_vp, _c_i64, _c_int,
                                          _c_vp, _c_vp, _c_i64]
        lib.oracle_gemm_mxfp8_entries.argtypes = [_c_i64, _c_dbl, _c_vp, _c_i64, _c_vp, _c_i64, _c_vp,
                                                  _c_i64, _c_vp, _c_i64, _c_dbl, _c_vp, _c_i64, _c_int,
                                                  _c_i64, _c_vp, _c_vp, _c_vp, _c_vp]
        lib.oracle_quantize_mxfp8.argtypes = [_c_i64, _c_i64, _c_vp, _c_i64, _c_vp, _c_i64, _c_vp, _c_i64]
        for fn in ("oracle_gemm", "oracle_gemm_entries", "oracle_syrk", "oracle_syrk_entries",
                   "oracle_syr2k", "oracle_syr2k_entries", "oracle_gemm_e4m3",
                   "oracle_gemm_e4m3_entries", "oracle_gemm_mxfp8", "oracle_gemm_mxfp8_entries",
                   "oracle_quantize_mxfp8"):
            getattr(lib, fn).restype = None
        self._lib = lib

    # -- helpers -------------------------------------------------------------
    @staticmethod
    def _bf16(x: np.ndarray) -> np.ndarray:
        x = np.ascontiguousarray(x)
        if x.dtype != np.uint16:
            raise TypeError("operands must be bf16 bit patterns (uint16)")
        return x

    @staticmethod
    def _cin(C, beta: float):
        """Returns (array or None, ld, is_bf16)."""
        if C is None:
            if beta != 0.0:
                raise ValueError("beta != 0 needs an input C")
            return None, 0, 0
        C = np.ascontiguousarray(C)
        if C.dtype == np.uint16:
            return C, C.shape[1], 1
        if C.dtype == np.float32:
            return C, C.shape[1], 0
        raise TypeError("C must be float32 or bf16 bit patterns (uint16)")

    @staticmethod
    def _ptr(a):
        return None if a is None else a.ctypes.data

    def num_threads(self) -> int:
        return int(self._lib.oracle_num_threads())

    def set_num_threads(self, n: int) -> None:
        """Threads of later calls (the results do not depend on it)."""
        self._lib.oracle_set_num_threads(int(n))

    # -- GEMM ----------------------------------------------------------------
    def gemm(self, m, n, k, transA, transB, alpha, A, B, beta=0.0, C=None):
        """Full m x n result (ref, bound) as float64 arrays.

        A is stored [m, k] (transA=0) or [k, m] (transA=1); B is [k, n] or
        [n, k]; the leading dimension is each array's row length.
        """
        A = self._bf16(A)
        B = self._bf16(B)
        Cin, ldc, cbf = self._cin(C, beta)
        ref = np.empty((m, n), dtype=np.float64)
        bound = np.empty((m, n), dtype=np.float64)
        self._lib.oracle_gemm(m, n, k, int(transA), int(transB), float(alpha),
                              A.ctypes.data, A.shape[1] if A.ndim == 2 else 0,
                              B.ctypes.data, B.shape[1] if B.ndim == 2 else 0,
                              float(beta), self._ptr(Cin), ldc, cbf,
                              ref.ctypes.data, bound.ctypes.data, n)
        return ref, bound

    def gemm_entries(self, k, transA, transB, alpha, A, B, rows, cols, beta=0.0, C=None):
        A = self._bf16(A)
        B = self._bf16(B)
        Cin, ldc, cbf = self._cin(C, beta)
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        cols = np.ascontiguousarray(cols, dtype=np.int64)
        ref = np.empty(rows.shape[0], dtype=np.float64)
        bound = np.empty(rows.shape[0], dtype=np.float64)
        self._lib.oracle_gemm_entries(k, int(transA), int(transB), float(alpha),
                                      A.ctypes.data, A.shape[1], B.ctypes.data, B.shape[1],
                                      float(beta), self._ptr(Cin), ldc, cbf, rows.shape[0],
                                      rows.ctypes.data, cols.ctypes.data,
                                      ref.ctypes.data, bound.ctypes.data)
        return ref, bound

    # -- SYRK ----------------------------------------------------------------
    def syrk(self, uplo, trans, n, k, alpha, A, beta=0.0, C=None):
        """Full n x n result; entries outside the triangle are NaN."""
        A = self._bf16(A)
        Cin, ldc, cbf = self._cin(C, beta)
        ref = np.empty((n, n), dtype=np.float64)
        bound = np.empty((n, n), dtype=np.float64)
        self._lib.oracle_syrk(int(uplo), int(trans), n, k, float(alpha), A.ctypes.data,
                              A.shape[1], float(beta), self._ptr(Cin), ldc, cbf,
                              ref.ctypes.data, bound.ctypes.data, n)
        return ref, bound

    def syrk_entries(self, uplo, trans, k, alpha, A, rows, cols, beta=0.0, C=None):
        A = self._bf16(A)
        Cin, ldc, cbf = self._cin(C, beta)
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        cols = np.ascontiguousarray(cols, dtype=np.int64)
        ref = np.empty(rows.shape[0], dtype=np.float64)
        bound = np.empty(rows.shape[0], dtype=np.float64)
        self._lib.oracle_syrk_entries(int(uplo), int(trans), k, float(alpha), A.ctypes.data,
                                      A.shape[1], float(beta), self._ptr(Cin), ldc, cbf,
                                      rows.shape[0], rows.ctypes.data, cols.ctypes.data,
                                      ref.ctypes.data, bound.ctypes.data)
        return ref, bound


    # -- GEMM with FP8 E4M3 operands --------------------------------------------
    @staticmethod
    def _e4m3(x: np.ndarray) -> np.ndarray:
        x = np.ascontiguousarray(x)
        if x.dtype != np.uint8:
            raise TypeError("operands must be E4M3 codes (uint8)")
        return x

    def gemm_e4m3(self, m, n, k, alpha, A, B, beta=0.0, C=None):
        """Full m x n result of alpha * A B^T + beta * C; A [m, k], B [n, k] E4M3 codes."""
        A = self._e4m3(A)
        B = self._e4m3(B)
        Cin, ldc, cbf = self._cin(C, beta)
        ref = np.empty((m, n), dtype=np.float64)
        bound = np.empty((m, n), dtype=np.float64)
        self._lib.oracle_gemm_e4m3(m, n, k, float(alpha), A.ctypes.data, A.shape[1], B.ctypes.data,
                                   B.shape[1], float(beta), self._ptr(Cin), ldc, cbf, ref.ctypes.data,
                                   bound.ctypes.data, n)
        return ref, bound

    def gemm_e4m3_entries(self, k, alpha, A, B, rows, cols, beta=0.0, C=None):
        A = self._e4m3(A)
        B = self._e4m3(B)
        Cin, ldc, cbf = self._cin(C, beta)
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        cols = np.ascontiguousarray(cols, dtype=np.int64)
        ref = np.empty(rows.shape[0], dtype=np.float64)
        bound = np.empty(rows.shape[0], dtype=np.float64)
        self._lib.oracle_gemm_e4m3_entries(k, float(alpha), A.ctypes.data, A.shape[1], B.ctypes.data,
                                           B.shape[1], float(beta), self._ptr(Cin), ldc, cbf, rows.shape[0],
                                           rows.ctypes.data, cols.ctypes.data, ref.ctypes.data,
                                           bound.ctypes.data)
        return ref, bound

    # -- GEMM with MXFP8 operands (E4M3 data, one UE8M0 scale per 32 along K) ---------
    @staticmethod
    def _scales(S, rows, k):
        S = np.ascontiguousarray(S)
        if S.dtype != np.uint8:
            raise TypeError("scales must be UE8M0 codes (uint8)")
        if S.shape[0] < rows or S.shape[1] < (k + 31) // 32:
            raise ValueError("scales must be [rows, >= ceil(k / 32)]")
        return S

    def gemm_mxfp8(self, m, n, k, alpha, A, SA, B, SB, beta=0.0, C=None):
        """Full m x n result of alpha * (A . SA)(B . SB)^T + beta * C.

        A [m, k] and B [n, k] hold E4M3 codes; SA [m, ceil(k/32)] and SB [n, ceil(k/32)]
        hold UE8M0 codes, row-major (each array's row length is its leading dimension).
        """
        A = self._e4m3(A)
        B = self._e4m3(B)
        SA = self._scales(SA, m, k)
        SB = self._scales(SB, n, k)
        Cin, ldc, cbf = self._cin(C, beta)
        ref = np.empty((m, n), dtype=np.float64)
        bound = np.empty((m, n), dtype=np.float64)
        self._lib.oracle_gemm_mxfp8(m, n, k, float(alpha), A.ctypes.data, A.shape[1], SA.ctypes.data,
                                    SA.shape[1], B.ctypes.data, B.shape[1], SB.ctypes.data, SB.shape[1],
                                    float(beta), self._ptr(Cin), ldc, cbf, ref.ctypes.data,
                                    bound.ctypes.data, n)
        return ref, bound

    def gemm_mxfp8_entries(self, k, alpha, A, SA, B, SB, rows, cols, beta=0.0, C=None):
        A = self._e4m3(A)
        B = self._e4m3(B)
        SA = self._scales(SA, 0, k)
        SB = self._scales(SB, 0, k)
        Cin, ldc, cbf = self._cin(C, beta)
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        cols = np.ascontiguousarray(cols, dtype=np.int64)
        ref = np.empty(rows.shape[0], dtype=np.float64)
        bound = np.empty(rows.shape[0], dtype=np.float64)
        self._lib.oracle_gemm_mxfp8_entries(k, float(alpha), A.ctypes.data, A.shape[1], SA.ctypes.data,
                                            SA.shape[1], B.ctypes.data, B.shape[1], SB.ctypes.data,
                                            SB.shape[1], float(beta), self._ptr(Cin), ldc, cbf,
                                            rows.shape[0], rows.ctypes.data, cols.ctypes.data,
                                            ref.ctypes.data, bound.ctypes.data)
        return ref, bound

    def quantize_mxfp8(self, X, k=None):
        """MXFP8 codes of the first k columns of a bf16 matrix X [rows, ld >= k] (k defaults
        to the row length): (E4M3 codes [rows, k], UE8M0 codes [rows, ceil(k/32)]), one
        scale per group of 32 along each row."""
        X = self._bf16(X)
        rows = X.shape[0]
        k = X.shape[1] if k is None else int(k)
        if not 0 <= k <= X.shape[1]:
            raise ValueError("k must be within the row length")
        Q = np.empty((rows, k), dtype=np.uint8)
        S = np.empty((rows, (k + 31) // 32), dtype=np.uint8)
        self._lib.oracle_quantize_mxfp8(rows, k, X.ctypes.data, X.shape[1], Q.ctypes.data, k,
                                        S.ctypes.data, S.shape[1])
        return Q, S

    # -- SYR2K ---------------------------------------------------------------
    def syr2k(self, uplo, trans, n, k, alpha, A, B, beta=0.0, C=None):
        """Full n x n result of alpha*(op(A) op(B)^T + op(B) op(A)^T) + beta*C; NaN off the triangle."""
        A = self._bf16(A)
        B = self._bf16(B)
        Cin, ldc, cbf = self._cin(C, beta)
        ref = np.empty((n, n), dtype=np.float64)
        bound = np.empty((n, n), dtype=np.float64)
        self._lib.oracle_syr2k(int(uplo), int(trans), n, k, float(alpha), A.ctypes.data, A.shape[1],
                               B.ctypes.data, B.shape[1], float(beta), self._ptr(Cin), ldc, cbf,
                               ref.ctypes.data, bound.ctypes.data, n)
        return ref, bound

    def syr2k_entries(self, uplo, trans, k, alpha, A, B, rows, cols, beta=0.0, C=None):
        A = self._bf16(A)
        B = self._bf16(B)
        Cin, ldc, cbf = self._cin(C, beta)
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        cols = np.ascontiguousarray(cols, dtype=np.int64)
        ref = np.empty(rows.shape[0], dtype=np.float64)
        bound = np.empty(rows.shape[0], dtype=np.float64)
        self._lib.oracle_syr2k_entries(int(uplo), int(trans), k, float(alpha), A.ctypes.data, A.shape[1],
                                       B.ctypes.data, B.shape[1], float(beta), self._ptr(Cin), ldc, cbf,
                                       rows.shape[0], rows.ctypes.data, cols.ctypes.data,
                                       ref.ctypes.data, bound.ctypes.data)
        return ref, bound


def build() -> str:
    """Compile the oracle if its shared object is missing or stale; returns its path."""
    with _lock:
        if _needs_build(_LIB_PATH, _SRC):
            compile_oracle()
    return _LIB_PATH


def default() -> Oracle:
    global _default
    if _default is None:
        _default = Oracle(build())
    return _default


# -- acceptance rule -----------------------------------------------------------
def tolerance(ref, bound, alpha, beta=0.0, c_in=None, out_bf16=False):
    """Per-element absolute tolerance of the acceptance rule in this module's docstring."""
    tol = 1e-3 * abs(float(alpha)) * np.asarray(bound, dtype=np.float64)
    if out_bf16:
        tol = tol + 2.0 ** -8 * np.abs(np.asarray(ref, dtype=np.float64))
    if c_in is not None and beta != 0.0:
        tol = tol + 2.0 ** -20 * np.abs(float(beta) * np.asarray(c_in, dtype=np.float64))
    return tol


def compare(got, ref, bound, alpha, beta=0.0, c_in=None, out_bf16=False):
    """Returns (ok, worst_ratio, index_of_worst); ratio = |got - ref| / tol (tol 0 -> exact)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    tol = tolerance(ref, bound, alpha, beta, c_in, out_bf16)
    err = np.abs(got - ref)
    bad_nan = np.isnan(got) != np.isnan(ref)
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = np.where(tol > 0, err / np.where(tol > 0, tol, 1.0), np.where(err > 0, np.inf, 0.0))
    ratio = np.where(np.isnan(ref) & np.isnan(got), 0.0, ratio)
    ratio = np.where(bad_nan, np.inf, ratio)
    if ratio.size == 0:
        return True, 0.0, None
    worst = int(np.nanargmax(ratio)) if not np.all(np.isnan(ratio)) else 0
    w = float(ratio.reshape(-1)[worst])
    return bool(w <= 1.0), w, np.unravel_index(worst, ratio.shape)
