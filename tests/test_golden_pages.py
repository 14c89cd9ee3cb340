"""The pages' printed 4096^3 timings pin the bench's flop accounting (CPU only).

Every row of tests/golden/pages_4096_timings.txt (page "cp.async / ldmatrix
ablation plan", section 0.3) satisfies TFLOP/s = 2*M*N*K / time to the printed
precision; a different convention (M*N*K, or 2*M*N*K with time in the wrong
unit) fails.
"""

import os

import bench

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "pages_4096_timings.txt")


def rows():
    out = []
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        name, prec, m, n, k, ms, tf = line.split()
        out.append((name, prec, int(m), int(n), int(k), float(ms), float(tf)))
    return out


def test_golden_rows_present():
    assert len(rows()) == 7


def test_flop_convention_matches_printed_throughput():
    for name, _, m, n, k, ms, tf in rows():
        got = bench.gemm_flops(m, n, k) / (ms * 1e-3) / 1e12
        assert abs(got - tf) <= 0.011, (name, got, tf)
        assert abs(m * n * k / (ms * 1e-3) / 1e12 - tf) > 1.0  # half the convention would not match


def test_pages_best_bf16_is_the_vs_baseline_reference():
    best = max(tf for _, prec, *_, tf in rows() if prec == "bf16")
    assert best == bench.PAGES_4096_TFLOPS


def test_work_accounting():
    assert bench.gemm_bytes(4096, 4096, 4096, 2, 0.0) == 3 * 4096 * 4096 * 2
    assert bench.gemm_bytes(5120, 5120, 2048, 2, 1.0) == 2 * (5120 * 2048 * 2) + 2 * 5120 * 5120 * 2
    assert bench.syrk_flops(8192, 4096) == 8192 * 8193 * 4096
    assert bench.syrk_bytes(8192, 4096, 4, 1.0) == 2 * 8192 * 4096 + 4 * (8192 * 8193 // 2) * 2
