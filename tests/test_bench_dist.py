"""The bench's multi-rank plumbing on CPU: two gloo ranks, no GPU.

The GEMM path does not shard: on N GPUs the bench runs N independent replicas,
and the only cross-rank traffic is a host barrier and the max over ranks of the
timed interval. These tests run that plumbing as two real processes over gloo
on 127.0.0.1, and the reference arm under torchrun, where rank 0 alone times
the oracle and prints the single JSON line while rank 1 exits 0 without work.
"""

import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), LOCAL_RANK=str(rank),
                      WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import bench
    d = bench.Dist()
    try:
        d.barrier()
        # each rank contributes a different interval; every rank must see the largest
        got = d.max(10.0 + 3.5 * rank)
        d.barrier()
        with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
            json.dump({"rank": d.rank, "world": d.world, "local": d.local, "max": got, "pg": d.pg}, f)
    finally:
        d.close()


def test_two_gloo_ranks_agree_on_the_max_interval(tmp_path):
    world = 2
    port = _free_port()
    mp.start_processes(_rank_main, args=(world, port, str(tmp_path)), nprocs=world, join=True,
                       start_method="spawn")
    results = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    for r, res in enumerate(results):
        assert res == {"rank": r, "world": world, "local": r, "max": 13.5, "pg": True}


def test_single_process_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    env = {k: os.environ.pop(k) for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK") if k in os.environ}
    try:
        d = bench.Dist()
        assert (d.world, d.rank, d.pg) == (1, 0, False)
        d.barrier()
        assert d.max(2.25) == 2.25
        d.close()
    finally:
        os.environ.update(env)


def test_reference_arm_under_torchrun_prints_one_line_from_rank_zero():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), "bench.py", "--impl", "reference",
           "--gpus", "2", "--steps", "3", "--warmup", "3", "--reference-budget-s", "1.5"]
    proc = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert proc.returncode == 0, proc.stderr[-2000:]
    lines = [ln for ln in proc.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, proc.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["steps"] == 3 and line["warmup"] == 3
    assert line["higher_is_better"] is True and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    # rank 0 runs alone, so it takes every host core rather than torchrun's one thread per rank
    assert line["cpu_baseline"]["cores"] == (os.cpu_count() or 1)
    assert line["e2e"] == {"value": line["value"], "unit": line["unit"], "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}
    assert line["config"]["workload"] == "gemm_bf16_4096x4096x4096_nn_bf16c"
