"""Seeded random GEMM calls that reach every launch plan, compared with the oracle on the
whole output.

Each case draws a shape from one of five families, chosen so that the planner takes a
different schedule for each: every tile split along K with a second kernel summing the
partials; a K split of the tail wave summed inside the kernel; the tail wave's tiles as
two half-column units; 128-row tiles on single SMs (short K or small outputs); whole
256 x 256 tiles on SM pairs. Transposes, alpha, beta, the C type and ragged edges are drawn
at random too. Operands and C hold small integers, so every product, partial sum and
combine is exact in FP32 and the whole output (and the guard band around it) must equal
the oracle's bit for bit. About half the cases round n down to a multiple of 8, so that
rows of C end on a 16-byte boundary and the epilogue stores C with TMA; the others store C
with masked plain stores.
"""

import random

import numpy as np
import pytest

import bm_inputs as gen
import oracle
from gpu_helpers import CBuffer, operand, run_gemm, torch

FAMILIES = ("all_split", "tail_k", "n_half", "single", "pair")


def _draw(rng, family):
    """(m, n, k, offer workspace) of one family; the tail families have 81 pair tiles (76 + 5)."""
    if family == "all_split":
        return rng.randint(1, 700), rng.randint(1, 700), rng.randint(2048, 5000), True
    if family == "tail_k":
        return rng.randint(2049, 2304), rng.randint(2049, 2304), rng.randint(2048, 2600), True
    if family == "n_half":
        return rng.randint(2049, 2304), rng.randint(2049, 2304), rng.randint(512, 1100), rng.random() < 0.5
    if family == "single":
        return rng.randint(1, 3000), rng.randint(1, 3000), rng.randint(1, 320), rng.random() < 0.5
    return rng.randint(2600, 3000), rng.randint(2600, 3000), rng.randint(384, 1000), rng.random() < 0.5


def _cases():
    rng = random.Random(0x5EED)
    out = []
    for rep in range(2):
        for family in FAMILIES:
            m, n, k, ws = _draw(rng, family)
            if n >= 8 and rng.random() < 0.5:  # rows of C that end on a 16-byte boundary take TMA stores
                n -= n % 8
            ta, tb = rng.randint(0, 1), rng.randint(0, 1)
            alpha = rng.choice([1.0, -1.0, 2.0])
            # a beta != 0 tail needs a larger gain to split along K: keep the K-split family at beta = 0
            beta = 0.0 if family == "tail_k" else rng.choice([0.0, 1.0, -1.0])
            bf16_out = rng.random() < 0.5
            out.append((family, m, n, k, ws, ta, tb, alpha, beta, bf16_out, 1000 + 10 * len(out)))
    return out


CASES = _cases()


def _branch(p):
    if p.kernels == 2:
        return "all_split"
    if p.k_splits > 1:
        return "tail_k"
    if p.n_splits == 2:
        return "n_half"
    return "single" if p.cta_pair == 1 else "pair"


@pytest.fixture(scope="module")
def lib():
    from blas3_tensor_core_gb300 import build
    build.build()


def test_cases_reach_every_plan(lib):
    """Host-only: the drawn cases take the schedule their family is meant to reach."""
    import blas3_tensor_core_gb300 as bm
    for family, m, n, k, ws, *_ in CASES:
        need = bm.bm_gemm_bf16_workspace_size(m, n, k) if ws else 0
        assert _branch(bm.bm_gemm_bf16_plan(m, n, k, need)[1]) == family, (family, m, n, k, ws)


@pytest.mark.gpu
@pytest.mark.parametrize("case", CASES, ids=[f"{c[0]}_{c[1]}x{c[2]}x{c[3]}" for c in CASES])
def test_random_plan_whole_output_exact(case, lib):
    import blas3_tensor_core_gb300 as bm
    t = torch()
    family, m, n, k, ws, ta, tb, alpha, beta, bf16_out, seed = case
    ra, ca = (k, m) if ta else (m, k)
    rb, cb = (n, k) if tb else (k, n)
    A = operand(ra, ca, "int", seed, lo=-3, hi=3, pad=8 - ca % 8)
    B = operand(rb, cb, "int", seed + 1, lo=-3, hi=3, pad=8 - cb % 8)
    c0 = gen.integers(seed + 2, m * n, -30, 30).reshape(m, n).astype(np.float32)
    c_init = gen.f32_to_bf16_bits(c0) if bf16_out else c0
    per = 8 if bf16_out else 4
    cbuf = CBuffer(m, n, n + (-n) % per + per, bf16_out, init=c_init)
    workspace = None
    if ws:
        need = bm.bm_gemm_bf16_workspace_size(m, n, k)
        workspace = t.full((max(need, 4) // 4,), float("nan"), dtype=t.float32, device="cuda")
    got, raw = run_gemm(m, n, k, ta, tb, alpha, A, B, beta, cbuf, workspace=workspace)
    cbuf.assert_guard_intact(raw)
    ref, _ = oracle.default().gemm(m, n, k, ta, tb, alpha, A, B, beta, c_init if beta != 0.0 else None)
    if bf16_out:
        ref = gen.bf16_bits_to_f32(gen.f32_to_bf16_bits(ref.astype(np.float32))).astype(np.float64)
    assert np.array_equal(got, ref), f"{family}: {int(np.sum(got != ref))} elements differ"
