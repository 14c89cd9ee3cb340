"""Seeded synthetic inputs for the BF16 GEMM / SYRK path.

This module is shared by the CPU oracle's tests, the GPU parity tests and the
bench. It holds none of the GEMM/SYRK arithmetic: only

* a counter-based generator (splitmix64, Steele/Lea/Flood 2014): element ``i``
  of the stream with seed ``s`` is ``mix(s + (i + 1) * 0x9E3779B97F4A7C15)``,
  so any block of a matrix can be regenerated without the rest;
* its mapping to uniform deviates in [0, 1) (top 53 bits) and to normal
  deviates by the Box-Muller transform (cosine branch, element ``i`` uses
  uniforms ``2i`` and ``2i+1``);
* IEEE round-to-nearest-even from float32 to bfloat16, and back;
* rounding from float32 to FP8 E4M3 (nearest, ties to even, saturating at
  448), and back, through the table of the format's 127 finite magnitudes.

The workloads are those of the BF16 GEMM shapes the pages study (square
4096^3, the K-sweep, the backward dX/dW pair and a lower SYRK): entries are
drawn in float64, rounded to float32, then to bfloat16 (round to nearest even
at both steps). Matrices are row-major NumPy arrays of bf16 bit patterns
(``uint16``) or float32.
"""

from __future__ import annotations

import numpy as np

__all__ = [
    "splitmix64",
    "uniform01",
    "uniform",
    "normal",
    "integers",
    "f32_to_bf16_bits",
    "bf16_bits_to_f32",
    "matrix_bf16",
    "matrix_f32",
    "symmetric_f32",
    "pad_ld",
    "BF16_NAN",
    "E4M3_VALUES",
    "f32_to_e4m3_bits",
    "e4m3_bits_to_f32",
    "matrix_e4m3",
]

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_MIX1 = np.uint64(0xBF58476D1CE4E5B9)
_MIX2 = np.uint64(0x94D049BB133111EB)
_TWO_PI = 2.0 * np.pi

BF16_NAN = np.uint16(0x7FC0)


def splitmix64(seed: int, index: np.ndarray) -> np.ndarray:
    """Counter-based splitmix64: one 64-bit word per element of ``index``."""
    idx = np.asarray(index, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + (idx + np.uint64(1)) * _GOLDEN
        z = (z ^ (z >> np.uint64(30))) * _MIX1
        z = (z ^ (z >> np.uint64(27))) * _MIX2
    return z ^ (z >> np.uint64(31))


def uniform01(seed: int, count: int, offset: int = 0) -> np.ndarray:
    """``count`` float64 deviates in [0, 1) from stream ``seed``, starting at ``offset``."""
    idx = np.arange(offset, offset + count, dtype=np.uint64)
    return (splitmix64(seed, idx) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def uniform(seed: int, count: int, lo: float, hi: float, offset: int = 0) -> np.ndarray:
    return lo + (hi - lo) * uniform01(seed, count, offset)


def normal(seed: int, count: int, std: float = 1.0, offset: int = 0) -> np.ndarray:
    """Box-Muller, cosine branch: element i uses uniforms 2i and 2i+1 of the stream."""
    idx = np.arange(offset, offset + count, dtype=np.uint64)
    u1 = (splitmix64(seed, 2 * idx) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)
    u2 = (splitmix64(seed, 2 * idx + np.uint64(1)) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)
    r = np.sqrt(-2.0 * np.log1p(-u1))  # 1 - u1 is in (0, 1]
    return std * r * np.cos(_TWO_PI * u2)


def integers(seed: int, count: int, lo: int, hi: int, offset: int = 0) -> np.ndarray:
    """Integers uniform in the closed range [lo, hi], as float64."""
    u = uniform01(seed, count, offset)
    return np.floor(u * (hi - lo + 1)) + lo


def f32_to_bf16_bits(x) -> np.ndarray:
    """Round float32 (float64 is first rounded to float32) to bfloat16, nearest-even."""
    f = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    u = f.view(np.uint32).astype(np.uint64)
    rounded = ((u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)).astype(np.uint16)
    return np.where(np.isnan(f), BF16_NAN, rounded).astype(np.uint16)


def bf16_bits_to_f32(b) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32."""
    u = np.ascontiguousarray(np.asarray(b, dtype=np.uint16)).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32)


def _draw(dist: str, seed: int, count: int, std: float, lo: float, hi: float) -> np.ndarray:
    if dist == "normal":
        return normal(seed, count, std)
    if dist == "uniform":
        return uniform(seed, count, lo, hi)
    if dist == "int":
        return integers(seed, count, int(lo), int(hi))
    raise ValueError(f"unknown distribution {dist!r}")


def matrix_bf16(rows: int, cols: int, dist: str = "normal", seed: int = 1, std: float = 1.0,
                lo: float = -1.0, hi: float = 1.0) -> np.ndarray:
    """Row-major [rows, cols] bf16 bit patterns; element (r, c) is stream index r*cols + c."""
    vals = _draw(dist, seed, rows * cols, std, lo, hi)
    return f32_to_bf16_bits(vals).reshape(rows, cols)


def matrix_f32(rows: int, cols: int, dist: str = "normal", seed: int = 3, std: float = 1.0,
               lo: float = -1.0, hi: float = 1.0) -> np.ndarray:
    vals = _draw(dist, seed, rows * cols, std, lo, hi)
    return vals.astype(np.float32).reshape(rows, cols)


def symmetric_f32(n: int, seed: int = 3, std: float = 1.0, dist: str = "normal",
                  lo: float = -1.0, hi: float = 1.0) -> np.ndarray:
    """Symmetric float32 [n, n]: the lower triangle is drawn, the upper mirrors it."""
    full = matrix_f32(n, n, dist, seed, std, lo, hi)
    low = np.tril(full)
    return (low + np.tril(full, -1).T).astype(np.float32)


def pad_ld(mat: np.ndarray, ld: int, fill) -> np.ndarray:
    """Copy a row-major matrix into rows of length ``ld`` (>= cols); the gap holds ``fill``."""
    rows, cols = mat.shape
    if ld < cols:
        raise ValueError("ld < cols")
    out = np.empty((rows, ld), dtype=mat.dtype)
    out[:, :cols] = mat
    out[:, cols:] = fill
    return out


# --- FP8 E4M3 (1 sign, 4 exponent bits with bias 7, 3 mantissa bits; no infinities;
# S.1111.111 is NaN; largest finite magnitude 448) -----------------------------------
def _e4m3_table() -> np.ndarray:
    """Value of every non-negative finite code 0x00..0x7E, in code order (increasing)."""
    vals = []
    for c in range(0x7F):
        e, m = c >> 3, c & 7
        vals.append((m / 8.0) * 2.0 ** -6 if e == 0 else (1.0 + m / 8.0) * 2.0 ** (e - 7))
    return np.array(vals, dtype=np.float64)


E4M3_VALUES = _e4m3_table()
E4M3_NAN = np.uint8(0x7F)


def f32_to_e4m3_bits(x) -> np.ndarray:
    """Round float32 values to E4M3: nearest representable value, ties to the even
    code, magnitudes beyond 448 saturate to 448, NaN stays NaN."""
    f = np.asarray(x, dtype=np.float32).astype(np.float64)
    a = np.abs(f)
    hi = np.clip(np.searchsorted(E4M3_VALUES, a, side="left"), 0, len(E4M3_VALUES) - 1)
    lo = np.clip(hi - 1, 0, len(E4M3_VALUES) - 1)
    d_hi = np.abs(E4M3_VALUES[hi] - a)
    d_lo = np.abs(a - E4M3_VALUES[lo])
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & ((hi & 1) == 0))
    code = np.where(pick_hi, hi, lo).astype(np.uint8)
    code = np.where(a >= E4M3_VALUES[-1], np.uint8(0x7E), code)  # saturate
    code = code | np.where(np.signbit(f), np.uint8(0x80), np.uint8(0))
    return np.where(np.isnan(f), E4M3_NAN, code).astype(np.uint8)


def e4m3_bits_to_f32(b) -> np.ndarray:
    b = np.asarray(b, dtype=np.uint8)
    mag = E4M3_VALUES[np.minimum(b & 0x7F, 0x7E)]
    out = np.where((b & 0x80) != 0, -mag, mag)
    return np.where((b & 0x7F) == 0x7F, np.nan, out).astype(np.float32)


def matrix_e4m3(rows: int, cols: int, dist: str = "normal", seed: int = 1, std: float = 1.0,
                lo: float = -1.0, hi: float = 1.0) -> np.ndarray:
    """Row-major [rows, cols] E4M3 codes (uint8); the value is drawn in float64, rounded to
    float32, then to E4M3 (nearest, ties to even, saturating)."""
    vals = _draw(dist, seed, rows * cols, std, lo, hi)
    return f32_to_e4m3_bits(vals.astype(np.float32)).reshape(rows, cols)
