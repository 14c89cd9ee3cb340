"""C-ABI library: loads, exports every declared symbol, validates arguments (CPU only).

No compute call reaches a GPU here: every call either fails argument checks
before any CUDA call, is a no-op (m == 0 or n == 0), or (on a machine without
a GPU) stops at the device query.
"""

import os
import re

import pytest

import blas3_tensor_core_gb300 as bm
from blas3_tensor_core_gb300 import build as bm_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    bm_build.build()
    return bm.library()


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "bm.h")).read()
    return sorted(set(re.findall(r"BM_API\s+[\w\s\*]*?\b(bm_\w+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_symbols()
    for required in ("bm_gemm_bf16", "bm_syrk_bf16", "bm_get_last_device_error", "bm_status_string"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    assert bm.bm_status_string(0) == "BM_OK"
    assert bm.bm_status_string(5) == "BM_ERR_TIMEOUT"
    assert bm.bm_status_string(99) == "BM_ERR_UNKNOWN"
    assert bm.bm_version() >= 100


def _gemm(m=64, n=64, k=64, ta=0, tb=0, A=0x1000, lda=None, B=0x2000, ldb=None, C=0x3000, ldc=None,
          ct=0, ws=None, wsb=0, alpha=1.0, beta=0.0):
    lda = lda if lda is not None else (m if ta else k)
    ldb = ldb if ldb is not None else (k if tb else n)
    ldc = ldc if ldc is not None else n
    return bm.bm_gemm_bf16(m, n, k, ta, tb, alpha, A, lda, B, ldb, beta, C, ldc, ct, ws, wsb, None)


def test_gemm_argument_errors(lib):
    assert _gemm(m=-1) == bm.BM_ERR_INVALID_VALUE
    assert _gemm(k=-5) == bm.BM_ERR_INVALID_VALUE
    assert _gemm(m=2 ** 31) == bm.BM_ERR_INVALID_VALUE
    assert _gemm(ta=2) == bm.BM_ERR_INVALID_VALUE
    assert _gemm(ct=7) == bm.BM_ERR_INVALID_VALUE
    assert _gemm(lda=63) == bm.BM_ERR_INVALID_VALUE              # lda < k
    assert _gemm(ta=1, lda=63) == bm.BM_ERR_INVALID_VALUE        # lda < m for op T
    assert _gemm(ldb=32) == bm.BM_ERR_INVALID_VALUE
    assert _gemm(ldc=60) == bm.BM_ERR_INVALID_VALUE
    assert _gemm(C=0) == bm.BM_ERR_INVALID_VALUE
    assert _gemm(A=0) == bm.BM_ERR_INVALID_VALUE
    assert _gemm(ws=None, wsb=1024) == bm.BM_ERR_WORKSPACE
    assert _gemm(ws=0x4010, wsb=1024) == bm.BM_ERR_WORKSPACE      # not 256-byte aligned


def test_gemm_alignment_errors(lib):
    assert _gemm(A=0x1008) == bm.BM_ERR_MISALIGNED
    assert _gemm(C=0x3004) == bm.BM_ERR_MISALIGNED
    assert _gemm(m=8, k=12, lda=12) == bm.BM_ERR_MISALIGNED       # 24-byte rows
    assert _gemm(n=10, ldc=10) == bm.BM_ERR_MISALIGNED            # fp32 C, 40-byte rows
    assert _gemm(n=12, ldc=12, ldb=16, ct=bm.BM_C_BF16) == bm.BM_ERR_MISALIGNED


def test_gemm_noops_touch_nothing(lib):
    assert _gemm(m=0) == bm.BM_OK
    assert _gemm(n=0, ldc=1, ldb=1) == bm.BM_OK


def test_alpha_zero_skips_operand_checks(lib):
    # A and B are not read when alpha == 0: their pointers may be null or misaligned.
    st = _gemm(alpha=0.0, A=0, B=0x2001)
    assert st != bm.BM_ERR_INVALID_VALUE and st != bm.BM_ERR_MISALIGNED


def test_syrk_split_plans(lib):
    """A triangle with too few tiles for the GPU is split along K when a workspace is given:
    n = 512, k = 8192 has 6 tiles of 128 x 256 (4 across the diagonal, 2 inside)."""
    for uplo in (bm.BM_LOWER, bm.BM_UPPER):
        assert bm.bm_syrk_bf16_plan(uplo, 512, 8192, 0)[1].k_splits == 1
        need = bm.bm_syrk_bf16_workspace_size(uplo, 512, 8192)
        p = bm.bm_syrk_bf16_plan(uplo, 512, 8192, need)[1]
        assert (p.tiles, p.cta_pair) == (6, 1)
        assert p.k_splits > 1 and p.kernels == 2 and p.split_tiles == 6
        assert p.workspace_bytes == need == p.k_splits * 6 * 128 * 256 * 4
        assert p.ctas <= 152 and p.ctas == min(152, 6 * p.k_splits)
    # SYR2K's k-blocks count both products
    assert bm.bm_syr2k_bf16_workspace_size(bm.BM_LOWER, 512, 4096) > 0
    assert bm.bm_syrk_bf16_workspace_size(bm.BM_LOWER, 512, 256) == 0      # too short to pay


def test_syrk_argument_errors(lib):
    def s(uplo=0, trans=0, n=64, k=64, A=0x1000, lda=None, C=0x3000, ldc=None, ct=0):
        lda = lda if lda is not None else (n if trans else k)
        ldc = ldc if ldc is not None else n
        return bm.bm_syrk_bf16(uplo, trans, n, k, 1.0, A, lda, 1.0, C, ldc, ct, None, 0, None)
    assert s(uplo=3) == bm.BM_ERR_INVALID_VALUE
    assert s(trans=5) == bm.BM_ERR_INVALID_VALUE
    assert s(n=-1) == bm.BM_ERR_INVALID_VALUE
    assert s(lda=10) == bm.BM_ERR_INVALID_VALUE
    assert s(trans=1, lda=32) == bm.BM_ERR_INVALID_VALUE
    assert s(ldc=32) == bm.BM_ERR_INVALID_VALUE
    assert s(A=0x1002) == bm.BM_ERR_MISALIGNED
    assert s(n=0, ldc=1) == bm.BM_OK
    assert bm.bm_syrk_bf16(0, 0, 64, 64, 1.0, 0x1000, 64, 1.0, 0x3000, 64, 0, None, 256, None) == bm.BM_ERR_WORKSPACE
    assert bm.bm_syrk_bf16(0, 0, 64, 64, 1.0, 0x1000, 64, 1.0, 0x3000, 64, 0, 0x4010, 256, None) \
        == bm.BM_ERR_WORKSPACE


def test_e4m3_argument_errors(lib):
    def g8(m=64, n=64, k=64, A=0x1000, lda=None, B=0x2000, ldb=None, C=0x3000, ldc=None, ct=0):
        lda = lda if lda is not None else k
        ldb = ldb if ldb is not None else k
        ldc = ldc if ldc is not None else n
        return bm.bm_gemm_e4m3(m, n, k, 1.0, A, lda, B, ldb, 0.0, C, ldc, ct, None, 0, None)
    assert g8(m=-1) == bm.BM_ERR_INVALID_VALUE
    assert g8(lda=32) == bm.BM_ERR_INVALID_VALUE     # lda < k
    assert g8(ldb=63) == bm.BM_ERR_INVALID_VALUE
    assert g8(k=72, lda=72, ldb=80) == bm.BM_ERR_MISALIGNED   # 72-byte rows
    assert g8(A=0x1008) == bm.BM_ERR_MISALIGNED
    assert g8(n=0, ldc=1) == bm.BM_OK
    assert bm.bm_gemm_e4m3_workspace_size(512, 512, 16384) > 0     # 128 k-blocks of 128: split pays
    # same bytes per k-block as bf16 with half the K (the lower beta == 0 tail-split threshold is
    # bf16-only, so compare where both split: a 16 us saving)
    assert bm.bm_gemm_e4m3_workspace_size(4096, 4096, 8192) == bm.bm_gemm_bf16_workspace_size(4096, 4096, 4096) > 0
    assert bm.bm_gemm_e4m3_workspace_size(4096, 4096, 4096) == 0    # 4.1 us: below the 6 us E4M3 keeps


def test_mxfp8_argument_errors_and_plans(lib):
    def g(m=64, n=64, k=64, A=0x1000, lda=None, SA=0x5000, B=0x2000, ldb=None, SB=0x6000, C=0x3000, ldc=None, ct=0):
        lda = lda if lda is not None else k
        ldb = ldb if ldb is not None else k
        ldc = ldc if ldc is not None else n
        return bm.bm_gemm_mxfp8(m, n, k, 1.0, A, lda, SA, B, ldb, SB, 0.0, C, ldc, ct, None, 0, None)
    assert g(m=-1) == bm.BM_ERR_INVALID_VALUE
    assert g(lda=32) == bm.BM_ERR_INVALID_VALUE
    assert g(SA=0) == bm.BM_ERR_INVALID_VALUE
    assert g(SB=0) == bm.BM_ERR_INVALID_VALUE
    assert g(SA=0x5008) == bm.BM_ERR_MISALIGNED
    assert g(k=72, lda=72, ldb=80) == bm.BM_ERR_MISALIGNED
    assert g(n=0, ldc=1) == bm.BM_OK
    # tiles 128 wide: 256 x 128 on SM pairs, 128 x 128 on single SMs; a k-block is 128 elements
    st, p = bm.bm_gemm_mxfp8_plan(4096, 4096, 4096, 0)
    assert st == 0 and (p.tile_m, p.tile_n, p.tile_k, p.cta_pair, p.tiles) == (256, 256, 128, 2, 16 * 16)
    assert (p.stages, p.stage_kblocks) == (5, 1)
    st, p = bm.bm_gemm_mxfp8_plan(1024, 2048, 4096, 0)   # 32 wide tiles: too few; 64 narrow ones fill
    assert (p.tile_m, p.tile_n, p.cta_pair, p.tiles) == (256, 128, 2, 64)
    st, p = bm.bm_gemm_mxfp8_plan(256, 256, 256, 0)
    assert (p.tile_m, p.tile_n, p.cta_pair, p.tiles) == (128, 128, 1, 4)
    assert bm.bm_gemm_mxfp8_workspace_size(512, 512, 16384) > 0
    # the scale-array size and the tiled layout's offsets
    assert bm.mxfp8_scale_bytes(129, 130) == 2 * 2 * 512
    assert bm.mxfp8_scale_offset(0, 0, 256) == 0
    assert bm.mxfp8_scale_offset(1, 0, 256) == 16 and bm.mxfp8_scale_offset(32, 0, 256) == 4
    assert bm.mxfp8_scale_offset(0, 1, 256) == 1 and bm.mxfp8_scale_offset(0, 4, 256) == 512
    assert bm.mxfp8_scale_offset(128, 0, 256) == 1024


def test_quantize_argument_errors(lib):
    def q(rows=64, k=64, X=0x1000, ldx=None, Q=0x2000, ldq=None, S=0x3000):
        ldx = ldx if ldx is not None else k
        ldq = ldq if ldq is not None else k
        return bm.bm_quantize_mxfp8(rows, k, X, ldx, Q, ldq, S, None)
    assert q(rows=-1) == bm.BM_ERR_INVALID_VALUE
    assert q(ldx=32) == bm.BM_ERR_INVALID_VALUE
    assert q(ldq=32) == bm.BM_ERR_INVALID_VALUE
    assert q(S=0) == bm.BM_ERR_INVALID_VALUE
    assert q(X=0x1008) == bm.BM_ERR_MISALIGNED
    assert q(k=36, ldx=36, ldq=48) == bm.BM_ERR_MISALIGNED       # 72-byte bf16 rows
    assert q(k=40, ldx=48, ldq=40) == bm.BM_ERR_MISALIGNED       # E4M3 rows not a multiple of 16
    assert q(S=0x3004) == bm.BM_ERR_MISALIGNED
    assert q(rows=0) == bm.BM_OK and q(k=0, ldx=1, ldq=1) == bm.BM_OK


def test_syr2k_argument_errors(lib):
    def s2(uplo=0, trans=0, n=64, k=64, A=0x1000, lda=None, B=0x2000, ldb=None, C=0x3000, ldc=None, ct=0):
        lda = lda if lda is not None else (n if trans else k)
        ldb = ldb if ldb is not None else (n if trans else k)
        ldc = ldc if ldc is not None else n
        return bm.bm_syr2k_bf16(uplo, trans, n, k, 1.0, A, lda, B, ldb, 1.0, C, ldc, ct, None, 0, None)
    assert s2(uplo=2) == bm.BM_ERR_INVALID_VALUE
    assert s2(trans=3) == bm.BM_ERR_INVALID_VALUE
    assert s2(k=-1) == bm.BM_ERR_INVALID_VALUE
    assert s2(ldb=10) == bm.BM_ERR_INVALID_VALUE
    assert s2(trans=1, lda=16) == bm.BM_ERR_INVALID_VALUE
    assert s2(B=0) == bm.BM_ERR_INVALID_VALUE
    assert s2(B=0x2004) == bm.BM_ERR_MISALIGNED
    assert s2(n=0, ldc=1) == bm.BM_OK


@pytest.mark.skipif(__import__("torch").cuda.is_available(), reason="expects a machine without a GPU")
def test_valid_call_without_gpu_reports_cuda_error(lib):
    assert _gemm() == bm.BM_ERR_CUDA


def test_gemm_plans(lib):
    # large outputs: 256 x 256 tiles on SM pairs, one CTA pair per SM pair
    st, p = bm.bm_gemm_bf16_plan(4096, 4096, 4096, 0)
    assert st == 0 and (p.tile_m, p.tile_n, p.tile_k, p.cta_pair) == (256, 256, 64, 2)
    assert p.tiles == 16 * 16 and p.k_splits == 1 and p.kernels == 1
    assert p.ctas == 152 and (p.stages, p.stage_kblocks) == (3, 2)  # 3 x 2 x 32 KB ring per CTA
    st, p = bm.bm_gemm_bf16_plan(2048, 5120, 5120, 0)
    assert p.tiles == 8 * 20 and p.cta_pair == 2
    # small outputs: 128-row tiles on single SMs
    st, p = bm.bm_gemm_bf16_plan(100, 100, 100, 0)
    assert p.tile_n == 128 and p.tiles == 1 and p.cta_pair == 1 and p.ctas == 1
    st, p = bm.bm_gemm_bf16_plan(512, 512, 256, 0)
    assert (p.tile_m, p.tile_n, p.cta_pair, p.tiles) == (128, 256, 1, 8)
    # a 512 x 512 output with K = 8192 fills the GPU only when K is split
    st, p = bm.bm_gemm_bf16_plan(512, 512, 8192, 0)
    assert p.k_splits == 1 and p.workspace_bytes == 0
    need = bm.bm_gemm_bf16_workspace_size(512, 512, 8192)
    assert need > 0
    st, p = bm.bm_gemm_bf16_plan(512, 512, 8192, need)
    # every tile split: the partial slots only, summed by the reduce kernel
    assert p.k_splits > 1 and p.kernels == 2 and p.workspace_bytes == need
    assert p.workspace_bytes == p.k_splits * 512 * 512 * 4
    st, p = bm.bm_gemm_bf16_plan(512, 512, 8192, need // 2)      # less workspace: fewer splits
    assert 1 <= p.k_splits < bm.bm_gemm_bf16_plan(512, 512, 8192, need)[1].k_splits
    assert p.workspace_bytes <= need // 2
    # short K: not worth a second kernel
    assert bm.bm_gemm_bf16_workspace_size(512, 512, 1024) == 0
    st, p = bm.bm_gemm_bf16_plan(64, 64, 0, 0)
    assert st == 0 and p.kernels == 1 and p.tiles == 0


def test_tail_split_plans(lib):
    # 4096^3 on SM pairs: 256 tiles = 3 full waves of 76 + 28; the 28 are split in two along K
    # and summed inside the kernel: two fp32 slots per split tile, then one 8-byte counter per
    # epilogue warp region (2 CTAs x 8 warps per tile); one kernel, no reduce launch
    need = bm.bm_gemm_bf16_workspace_size(4096, 4096, 4096)
    assert need == 2 * 28 * 256 * 256 * 4 + 28 * 2 * 8 * 8
    p = bm.bm_gemm_bf16_plan(4096, 4096, 4096, need)[1]
    assert (p.split_tiles, p.k_splits, p.kernels, p.ctas) == (28, 2, 1, 152)
    # one byte short of the counters: no K split
    assert bm.bm_gemm_bf16_plan(4096, 4096, 4096, need - 1)[1].k_splits == 1
    # no workspace: no K split; the 28 tail tiles run as two halves of their columns each
    # (no partial sums, so no workspace), on 56 SM pairs
    p = bm.bm_gemm_bf16_plan(4096, 4096, 4096, 0)[1]
    assert (p.split_tiles, p.k_splits, p.n_splits, p.kernels, p.workspace_bytes) == (28, 1, 2, 1, 0)
    # dX 2048x5120x5120: 160 tiles = 2 waves + 8; split 7 ways within the 16 MiB tail budget
    # (8 ways would need 16 MiB of slots plus the counters)
    p = bm.bm_gemm_bf16_plan(2048, 5120, 5120, 1 << 30)[1]
    assert (p.split_tiles, p.k_splits, p.kernels) == (8, 7, 1) and p.workspace_bytes <= 16 << 20
    # the tail split must save enough mainloop time: 3.5 us for a beta == 0 bf16 GEMM (the
    # plan shown), 6 us with beta != 0; 0.256 us per k-block of a tile
    p = bm.bm_gemm_bf16_plan(5120, 5120, 2048, 1 << 30)[1]     # 400 tiles = 5 waves + 20
    assert (p.split_tiles, p.k_splits) == (20, 3)              # 3-way: 21 of 32 k-blocks saved, 5.4 us
    p = bm.bm_gemm_bf16_plan(5120, 5120, 4096, 1 << 30)[1]
    assert p.split_tiles == 20 and p.k_splits == 3
    p = bm.bm_gemm_bf16_plan(4096, 4096, 1024, 1 << 30)[1]     # 2-way: 8 k-blocks, 2 us: no K split,
    assert (p.split_tiles, p.k_splits, p.n_splits) == (28, 1, 2)  # N halves instead
    p = bm.bm_gemm_bf16_plan(4096, 4096, 2048, 1 << 30)[1]     # 2-way: 16 k-blocks, 4.1 us
    assert (p.split_tiles, p.k_splits, p.n_splits) == (28, 2, 1)
    # N halves are for 256 x 256 bf16 pair tiles only: single-SM tiles (short K) and E4M3 keep
    # whole tail tiles
    p = bm.bm_gemm_bf16_plan(4096, 4096, 256, 1 << 30)[1]
    assert p.cta_pair == 1 and p.n_splits == 1
    # a last wave more than half full is not split
    p = bm.bm_gemm_bf16_plan(8192, 8192 - 1024, 4096, 1 << 30)[1]  # 32 x 28 = 896 tiles = 11 waves + 60
    assert p.split_tiles == 0 and p.k_splits == 1
    # SYRK 8192 x 4096: 528 pair tiles = 6 waves + 72, a last wave more than half full
    assert bm.bm_syrk_bf16_plan(bm.BM_LOWER, 8192, 4096, 1 << 30)[1].k_splits == 1
    assert bm.bm_gemm_bf16_plan(-1, 4, 4, 0)[0] == bm.BM_ERR_INVALID_VALUE


def _syrk_tiles_bruteforce(n, lower, bm_=128, bn=256):
    tiles = 0
    for tm in range((n + bm_ - 1) // bm_):
        for tn in range((n + bn - 1) // bn):
            rows = range(tm * bm_, min(n, tm * bm_ + bm_))
            cols = range(tn * bn, min(n, tn * bn + bn))
            # does the tile hold an element of the triangle (nominal tile extents)?
            r_lo, r_hi, c_lo, c_hi = tm * bm_, tm * bm_ + bm_ - 1, tn * bn, tn * bn + bn - 1
            if (lower and r_hi >= c_lo) or (not lower and r_lo <= c_hi):
                tiles += 1
                assert rows and cols
    return tiles


@pytest.mark.parametrize("n", [1, 100, 128, 129, 256, 300, 1000, 8192])
def test_syrk_plans_visit_only_triangle_tiles(lib, n):
    for uplo in (bm.BM_LOWER, bm.BM_UPPER):
        st, p = bm.bm_syrk_bf16_plan(uplo, n, 64)
        assert st == 0
        assert p.tiles == _syrk_tiles_bruteforce(n, uplo == bm.BM_LOWER, p.tile_m, p.tile_n)
    if n == 8192:
        # 32 x 32 square tiles of 256 on SM pairs: 32 * 33 / 2 on or below the diagonal
        p = bm.bm_syrk_bf16_plan(bm.BM_LOWER, n, 64)[1]
        assert (p.tile_m, p.tile_n, p.cta_pair, p.tiles) == (256, 256, 2, 528)
    if n <= 256:
        assert bm.bm_syrk_bf16_plan(bm.BM_LOWER, n, 64)[1].cta_pair == 1


def test_tile_override_values(lib):
    assert bm.bm_set_tile_override(5) == bm.BM_ERR_INVALID_VALUE
    assert bm.bm_set_tile_override(-1) == bm.BM_ERR_INVALID_VALUE
    try:
        for v, want in [(1, (128, 256, 1)), (2, (128, 128, 1)), (3, (256, 256, 2))]:
            assert bm.bm_set_tile_override(v) == bm.BM_OK
            p = bm.bm_gemm_bf16_plan(1000, 1000, 64, 0)[1]
            assert (p.tile_m, p.tile_n, p.cta_pair) == want
            s = bm.bm_syrk_bf16_plan(bm.BM_LOWER, 1000, 64)[1]
            assert (s.tile_m, s.tile_n, s.cta_pair) == want
            assert s.tiles == _syrk_tiles_bruteforce(1000, True, s.tile_m, s.tile_n)
    finally:
        assert bm.bm_set_tile_override(0) == bm.BM_OK


def _syrk_order_bruteforce(n, lower, tm_, tn_, group=16):
    """The schedule written out by enumeration: per tile row the tile that crosses the
    diagonal, then the tiles wholly inside the triangle (nominal tile extents). Inside
    tiles: with square tiles, groups of `group` tile rows of the lower triangle, each
    column by column (rows in order within a column), and for the upper triangle the
    transpose of that; with 128 x 256 tiles, row by row."""
    rows_t, cols_t = (n + tm_ - 1) // tm_, (n + tn_ - 1) // tn_
    cross, inside = [], []
    for r in range(rows_t):
        for c in range(cols_t):
            r_lo, r_hi, c_lo, c_hi = r * tm_, r * tm_ + tm_ - 1, c * tn_, c * tn_ + tn_ - 1
            touches = r_hi >= c_lo if lower else r_lo <= c_hi
            wholly = r_lo >= c_hi if lower else r_hi <= c_lo
            if touches and wholly:
                inside.append((r, c))
            elif touches:
                cross.append((r, c))
    if tm_ == tn_:
        members = set(inside)
        grouped = []
        for r0 in range(0, rows_t, group):
            r1 = min(r0 + group, rows_t)
            for c in range(cols_t):
                for r in range(r0, r1):
                    t = (r, c) if lower else (c, r)
                    if t in members:
                        grouped.append(t)
        assert sorted(grouped) == sorted(inside)
        inside = grouped
    return cross + inside


@pytest.mark.parametrize("n", [1, 200, 256, 300, 1000, 1024, 2200, 4096, 4352, 8192, 12288 + 100, 16384, 33000])
@pytest.mark.parametrize("variant", [1, 2, 3], ids=["single128x256", "single128x128", "pair256x256"])
def test_syrk_tile_order_closed_form(lib, n, variant):
    """Every tile index of the kernel's closed-form SYRK schedule maps to the tile the
    enumeration puts there: the diagonal-crossing tiles first, then the inside ones
    (grouped for square tiles). Sizes cover one group, a partial last group (including
    one of a single tile row) and many groups."""
    import numpy as np
    assert bm.bm_set_tile_override(variant) == bm.BM_OK
    try:
        for uplo in (bm.BM_LOWER, bm.BM_UPPER):
            st, p = bm.bm_syrk_bf16_plan(uplo, n, 64)
            assert st == 0
            want = _syrk_order_bruteforce(n, uplo == bm.BM_LOWER, p.tile_m, p.tile_n)
            st, rows, cols = bm.bm_syrk_bf16_tile_order(uplo, n, 64)
            assert st == 0 and p.tiles == len(want)
            got = list(zip(rows.tolist(), cols.tolist()))
            assert got == want
            # one tile across the diagonal per tile row, in row order
            tiles_m = (n + p.tile_m - 1) // p.tile_m
            assert [r for r, _ in want[:tiles_m]] == list(range(tiles_m))
    finally:
        bm.bm_set_tile_override(0)


def test_syrk_tile_order_argument_errors(lib):
    import ctypes
    import numpy as np
    st, p = bm.bm_syrk_bf16_plan(bm.BM_LOWER, 1000, 64)
    buf = np.zeros(p.tiles + 1, np.int64)
    f = bm.library().bm_syrk_bf16_tile_order
    assert f(bm.BM_LOWER, 1000, 64, p.tiles + 1, buf.ctypes.data, buf.ctypes.data) == bm.BM_ERR_INVALID_VALUE
    assert f(bm.BM_LOWER, 1000, 64, p.tiles, None, None) == bm.BM_ERR_INVALID_VALUE
    assert f(7, 1000, 64, p.tiles, buf.ctypes.data, buf.ctypes.data) == bm.BM_ERR_INVALID_VALUE
    assert f(bm.BM_LOWER, 0, 64, 0, None, None) == bm.BM_OK


def test_short_k_bf16_gemms_plan_single_sm_tiles(lib):
    """BF16 GEMMs of at most five 64-deep k-blocks (K <= 320) take 128 x 256 single-SM
    tiles; from six k-blocks on, outputs that fill half the SM pairs take 256 x 256 pairs."""
    for m, n, k in [(4096, 4096, 256), (4096, 4096, 320), (8192, 8192, 256), (2048, 2048, 64)]:
        p = bm.bm_gemm_bf16_plan(m, n, k, 0)[1]
        assert (p.tile_m, p.tile_n, p.cta_pair) == (128, 256, 1), (m, n, k)
    for m, n, k in [(4096, 4096, 384), (4096, 4096, 512), (8192, 8192, 512)]:
        p = bm.bm_gemm_bf16_plan(m, n, k, 0)[1]
        assert (p.tile_m, p.tile_n, p.cta_pair) == (256, 256, 2), (m, n, k)


def test_full_splits_capped_at_14_ways(lib):
    """Every tile of a small output is split along K at most 14 ways: 512^2 x 8192 and
    x 4096 split their 8 tiles 13 ways; SYRK 512 x 8192 its 6 tiles 13 ways."""
    for k in (4096, 8192):
        need = bm.bm_gemm_bf16_workspace_size(512, 512, k)
        p = bm.bm_gemm_bf16_plan(512, 512, k, need)[1]
        assert p.tiles == 8 and p.k_splits == 13 and p.kernels == 2, k
    for uplo in (bm.BM_LOWER, bm.BM_UPPER):
        need = bm.bm_syrk_bf16_workspace_size(uplo, 512, 8192)
        p = bm.bm_syrk_bf16_plan(uplo, 512, 8192, need)[1]
        assert p.tiles == 6 and p.k_splits == 13 and p.kernels == 2


def _cdiv(a, b):
    return -(-a // b)


def _check_plan(p, m, n, k, budget, kblock, pair_slots=76, sms=152, tiles=None):
    """Invariants every plan keeps, whatever the shape and the workspace offered (tiles: the
    expected tile count where it is not the whole m x n grid)."""
    assert p.tiles == (tiles if tiles is not None else _cdiv(m, p.tile_m) * _cdiv(n, p.tile_n))
    assert p.cta_pair in (1, 2) and (p.cta_pair == 1 or p.tile_m == 256)
    assert 0 <= p.split_tiles <= p.tiles and p.k_splits >= 1 and p.n_splits in (1, 2)
    kb = _cdiv(k, kblock)
    if p.k_splits > 1:
        per = _cdiv(kb, p.k_splits)
        assert per >= 4 and _cdiv(kb, per) == p.k_splits      # every part keeps >= 4 k-blocks, none empty
        assert 0 < p.workspace_bytes <= budget
        assert p.n_splits == 1
        if p.kernels == 2:                                      # every tile split, summed by a second kernel
            assert p.split_tiles == p.tiles and p.k_splits <= 14
            assert p.workspace_bytes == p.k_splits * p.tiles * p.tile_m * p.tile_n * 4
        else:                                                   # a tail split, summed inside the kernel
            assert p.kernels == 1 and 0 < p.split_tiles < p.tiles
            assert p.workspace_bytes <= 16 << 20
    else:
        assert p.workspace_bytes == 0 and p.kernels == 1
    if p.n_splits == 2:                                         # tail tiles as two N halves: no partials
        assert (p.cta_pair, p.tile_n, p.k_splits, p.workspace_bytes) == (2, 256, 1, 0)
        assert 0 < p.split_tiles and p.split_tiles * 2 <= pair_slots
    if p.k_splits == 1 and p.n_splits == 1:
        assert p.split_tiles == 0
    slots = pair_slots if p.cta_pair == 2 else sms
    if 0 < p.split_tiles < p.tiles:                             # only an at most half-full last wave
        assert p.split_tiles == p.tiles % slots and p.split_tiles * 2 <= slots
    units = p.tiles - p.split_tiles + p.split_tiles * max(p.k_splits, p.n_splits)
    assert p.ctas == (2 * min(units, pair_slots) if p.cta_pair == 2 else min(units, sms))


def test_gemm_plan_invariants_over_random_shapes(lib):
    """Seeded random shapes (sizes from 1 to 16384, K up to 32768) and workspace offers:
    tile counts, split bounds, workspace sizes, half-column units and the grid agree with
    the planning rules, and the size query returns what an unlimited offer plans."""
    import random
    rng = random.Random(20240611)
    dims = [1, 7, 64, 100, 128, 129, 255, 256, 257, 511, 512, 1000, 1024, 2048, 3000, 4096, 5120, 8192, 16384]
    for _ in range(400):
        m, n = rng.choice(dims), rng.choice(dims)
        k = rng.choice([1, 63, 64, 256, 320, 384, 512, 1024, 2048, 4096, 5000, 8192, 32768])
        need = bm.bm_gemm_bf16_workspace_size(m, n, k)
        unlimited = bm.bm_gemm_bf16_plan(m, n, k, 1 << 40)[1]
        assert need == unlimited.workspace_bytes
        for budget in (0, need // 2, need, 1 << 40):
            st, p = bm.bm_gemm_bf16_plan(m, n, k, budget)
            assert st == 0
            _check_plan(p, m, n, k, budget, 64)
            if budget >= need:                                  # enough workspace: the same plan
                assert (p.k_splits, p.split_tiles, p.n_splits) == (unlimited.k_splits, unlimited.split_tiles,
                                                                   unlimited.n_splits)
        p0 = bm.bm_gemm_bf16_plan(m, n, k, 0)[1]
        assert p0.k_splits == 1 and p0.workspace_bytes == 0


def test_mxfp8_and_syrk_plan_invariants_over_random_shapes(lib):
    """The same invariants for MXFP8 GEMM plans (128-deep k-blocks, no half-column units) and
    for SYRK plans (only the triangle's tiles, counted by enumeration)."""
    import random
    rng = random.Random(7)
    dims = [1, 100, 128, 129, 256, 300, 512, 1000, 2048, 4096, 8192]
    for _ in range(150):
        m, n = rng.choice(dims), rng.choice(dims)
        k = rng.choice([32, 128, 512, 1024, 4096, 8192, 32768])
        need = bm.bm_gemm_mxfp8_workspace_size(m, n, k)
        for budget in (0, need // 2, need, 1 << 40):
            st, p = bm.bm_gemm_mxfp8_plan(m, n, k, budget)
            assert st == 0 and p.tile_k == 128 and p.n_splits == 1
            assert (p.tile_m, p.tile_n, p.cta_pair) in ((256, 256, 2), (256, 128, 2), (128, 128, 1))
            _check_plan(p, m, n, k, budget, 128)
    for n in (1, 100, 256, 300, 513, 1000, 2048, 4100, 8192):
        for k in (64, 512, 4096, 8192, 32768):
            for uplo in (bm.BM_LOWER, bm.BM_UPPER):
                need = bm.bm_syrk_bf16_workspace_size(uplo, n, k)
                for budget in (0, need, 1 << 40):
                    st, p = bm.bm_syrk_bf16_plan(uplo, n, k, budget)
                    assert st == 0 and p.n_splits == 1
                    expect = _syrk_tiles_bruteforce(n, uplo == bm.BM_LOWER, p.tile_m, p.tile_n)
                    _check_plan(p, n, n, k, budget, 64, tiles=expect)


def test_tensor_helpers_reject_bad_arguments_before_any_call():
    """The torch-tensor helpers check dtype, shapes, layout and device before they reach the
    C ABI: a host tensor's address must never be passed on as a device pointer."""
    import torch
    bf, f32 = torch.bfloat16, torch.float32
    A, B, C = torch.zeros(4, 8, dtype=bf), torch.zeros(8, 6, dtype=bf), torch.zeros(4, 6, dtype=f32)
    with pytest.raises(ValueError, match="CUDA tensor"):
        bm.gemm(A, B, C)
    with pytest.raises(TypeError):
        bm.gemm(A.float(), B, C)
    with pytest.raises(TypeError):
        bm._ctype(C.to(torch.float16))
    with pytest.raises(ValueError, match="inconsistent"):
        bm.gemm(A, B, torch.zeros(4, 7, dtype=f32))
    with pytest.raises(ValueError, match="inconsistent"):
        bm.gemm(A, B, C, transA=True)
    with pytest.raises(ValueError, match="CUDA tensor"):
        bm.gemm(A.t().contiguous(), B.t().contiguous(), C, transA=True, transB=True)
    with pytest.raises(ValueError, match="row-major"):
        bm._rowmajor_ld(C.t(), "C")
    assert bm._rowmajor_ld(C, "C") == 6 and bm._rowmajor_ld(torch.zeros(3, 10)[:, :6], "C") == 10
    S = torch.zeros(4, 4, dtype=f32)
    with pytest.raises(ValueError, match="CUDA tensor"):
        bm.syrk(A, S)
    with pytest.raises(ValueError, match="square"):
        bm.syrk(A, C)
    with pytest.raises(ValueError, match="inconsistent"):
        bm.syrk(A, S, trans=True)
    with pytest.raises(ValueError, match="same shape"):
        bm.syr2k(A, B, S)
    with pytest.raises(ValueError, match="CUDA tensor"):
        bm.syr2k(A, A.clone(), S)
