"""Host-side bench logic that needs no GPU: the source hash that ties a committed
ncu summary to the kernel code it was taken on."""

import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _write(d, text):
    d.mkdir(exist_ok=True)
    (d / "k.cuh").write_text(text)
    return str(d)


def test_source_hash_ignores_comments_and_whitespace(tmp_path):
    import bench
    base = "int f(int x)\n{\n    return x + 1;  // one more\n}\n"
    same = "/* header\n   comment */\nint f(int x) {\n  return   x + 1;\n}\n// trailing\n"
    other = "int f(int x)\n{\n    return x + 2;  // one more\n}\n"
    h0 = bench.kernel_source_hash(_write(tmp_path / "a", base))
    assert bench.kernel_source_hash(_write(tmp_path / "b", same)) == h0
    assert bench.kernel_source_hash(_write(tmp_path / "c", other)) != h0


def test_committed_summary_names_its_hash_and_traffic():
    import bench
    text = open(os.path.join(ROOT, "profiles", "gemm_bf16_4096x4096x4096_nn_bf16c.ncu.txt")).read()
    fields = dict(line.split(":", 1) for line in text.splitlines() if ":" in line and not line.startswith(" "))
    assert len(fields["kernel_source_sha256"].strip()) == 64
    assert float(fields["dram_bytes_per_launch"]) > 100e6  # at least the algorithmic 100.7 MB of a 4096^3 call


def test_percentiles_interpolate_between_order_statistics():
    import bench
    v = [5.0, 1.0, 3.0, 2.0, 4.0]
    assert bench.percentile(v, 0) == 1.0 and bench.percentile(v, 100) == 5.0
    assert bench.percentile(v, 50) == 3.0
    assert abs(bench.percentile(v, 95) - 4.8) < 1e-12
    assert bench.percentile([7.0], 95) == 7.0


def test_config_list_covers_every_configured_workload():
    """C1 256^3, C2 4096^3, the ten sweep shapes, both backward GEMMs and the SYRK, each once."""
    import bench
    labels = [lab for lab, _ in bench.CONFIG_ORDER]
    names = [c["name"] for _, c in bench.CONFIG_ORDER]
    assert len(set(names)) == len(names)
    assert labels.count("C1") == 1 and labels.count("C2") == 1 and labels.count("C3") == 10
    assert labels.count("C4a") == labels.count("C4b") == labels.count("C5") == 1
    sweep = {(c["m"], c["k"]) for lab, c in bench.CONFIG_ORDER if lab == "C3"}
    assert sweep == {(mn, k) for mn in (512, 4096) for k in (256, 512, 1024, 4096, 8192)}
    dw = dict(bench.CONFIG_ORDER)["C4b"]
    assert (dw["m"], dw["n"], dw["k"], dw["ta"], dw["beta"], dw["std"]) == (5120, 5120, 2048, 1, 1.0, 0.02)
    assert dict(bench.CONFIG_ORDER)["C5"]["n"] == 8192 and dict(bench.CONFIG_ORDER)["C5"]["k"] == 4096


def test_both_arms_share_the_config_dict():
    import bench
    assert bench.main_config() == bench.main_config()
    assert bench.main_config()["workload"] == bench.MAIN["name"]
    # nothing run-specific (L2 sets, plan) inside it: those live beside it in the GPU line
    assert not {"l2", "plan"} & set(bench.main_config())


class _FakeWorkload:
    """Stands in for a configured workload: fixed flops and bytes, an optional plan."""

    def __init__(self, flops, nbytes, plan=None, e4m3=False):
        self.name, self._f, self._b, self.plan, self.e4m3 = "fake", flops, nbytes, plan, e4m3

    def flops(self):
        return self._f

    def bytes(self):
        return self._b

    def tensor_peak(self, peaks):
        return peaks["bf16_tflops"]

    def kind(self):
        return "gemm"

    def flop_convention(self):
        return "2mnk"


def test_config_record_bound_fractions_and_plan():
    """The bound is whichever peak the workload would take longer at; the fraction is taken against
    that peak; the plan is copied field by field, with a note on the E4M3 stand-in and none without a plan."""
    import types
    import bench
    peaks = {"bf16_tflops": 2000.0, "hbm_gbs": 8000.0}
    stats = {"p50": 0.1, "p95": 0.12, "min": 0.09, "mean": 0.1, "n": 20}  # ms
    keys = ("tile_m", "tile_n", "cta_pair", "tiles", "k_splits", "n_splits", "split_tiles", "kernels", "ctas")
    plan = types.SimpleNamespace(**{k: i + 1 for i, k in enumerate(keys)})

    dense = bench.config_record("C2", _FakeWorkload(1e11, 1e5, plan), stats, peaks, 0.08, 0.07)
    assert dense["bound"] == "tensor"
    assert abs(dense["tflops_p50"] - 1000.0) < 1e-9 and dense["roofline_frac_p50"] == 0.5
    assert dense["roofline_frac_back_to_back"] == 0.625 and dense["us_per_call_graph"] == 70.0
    assert dense["plan"] == {k: i + 1 for i, k in enumerate(keys)}

    streaming = bench.config_record("C3", _FakeWorkload(1e9, 4e8, None), stats, peaks, 0.1, 0.1)
    assert streaming["bound"] == "hbm" and streaming["plan"] == {}
    assert abs(streaming["gbs_p50"] - 4000.0) < 1e-9 and streaming["roofline_frac_p50"] == 0.5

    fp8 = bench.config_record("F8", _FakeWorkload(1e11, 1e5, plan, e4m3=True), stats, peaks, 0.08, 0.07)
    assert "K/2" in fp8["plan"]["note"]


def test_cpu_baseline_sample_is_sized_and_bounded():
    """The oracle sample of the CPU baseline: calibrated on a probe, capped at the whole
    matrix, and its rows equal the oracle's full result for those rows."""
    import numpy as np
    import bm_inputs as gen
    import bench
    import oracle
    cfg = dict(bench.MAIN, m=96, n=64, k=128)
    A = gen.matrix_bf16(96, 128, "normal", 1)
    B = gen.matrix_bf16(128, 64, "normal", 2)
    r = bench.oracle_rows_rate(A, B, cfg, budget_s=60.0)        # a tiny matrix: the whole of it
    assert r["rows"] == 96 and r["ref"].shape == (96, 64) and r["tflops"] > 0 and r["cores"] >= 1
    full, _ = oracle.default().gemm(96, 64, 128, 0, 0, 1.0, A, B)
    assert np.array_equal(r["ref"], full)
    r = bench.oracle_rows_rate(A, B, cfg, budget_s=1e-6)         # no budget: the minimum sample
    assert r["rows"] == 4
