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
