"""bench.py's multi-GPU path on the CPU: two replica ranks over gloo.

`bench.py --gpus N` under torchrun runs one independent replica per GPU (the
path needs no exchange); the whole-job value is the work of all ranks over
the slowest rank's time.  Here two processes with different timed totals
reduce through `replica_throughput` over a gloo process group, and the
reference arm's non-zero ranks leave without work."""

import json
import multiprocessing as mp
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, totals, out_q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        assert bench.dist_info() == (rank, world, rank)
        vals, maxed = bench.replica_throughput(torch, world, 2.0e12, 10, totals[rank])
        out_q.put((rank, vals, maxed))
    finally:
        dist.destroy_process_group()


def test_two_replicas_take_the_slowest_rank():
    world, port = 2, _free_port()
    totals = {0: [100.0, 400.0], 1: [125.0, 300.0]}  # ms: step total, e2e total
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, totals, q)) for r in range(world)]
    for p in procs:
        p.start()
    results = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, vals, maxed in results:
        assert maxed == [125.0, 400.0]
        # 2 ranks x 10 steps x 2 TFLOP over the slowest rank's 0.125 s / 0.4 s
        assert vals == pytest.approx([2 * 10 * 2.0 / 0.125, 2 * 10 * 2.0 / 0.4])


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import torch
    import bench
    vals, maxed = bench.replica_throughput(torch, 1, 1.0e12, 4, [200.0])
    assert maxed == [200.0] and vals == pytest.approx([4 * 1.0 / 0.2])


def test_reference_arm_other_ranks_exit_without_work(tmp_path):
    import subprocess
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3"], env=env, capture_output=True, text=True,
                       timeout=300, cwd=str(tmp_path))
    assert r.returncode == 0
    assert r.stdout.strip() == ""


def test_reference_arm_line_carries_the_contract_keys(tmp_path):
    """The reference arm (the float64 oracle on the host cores) prints one JSON
    line with the keys the bench contract names, on the headline workload."""
    import json
    import subprocess
    env = {k: v for k, v in os.environ.items() if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK")}
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3"], env=env, capture_output=True, text=True,
                       timeout=600, cwd=str(tmp_path))
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["steps"] == 1 and d["warmup"] == 3
    assert d["value"] > 0 and d["higher_is_better"] is True
    assert d["config"]["workload"] == "llama3_8b_sft_packing_gqa32x8_d128_t8192"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["sample"]
    assert cb["value"] == d["value"]
    e = d["e2e"]
    assert e["value"] == d["value"] and e["unit"] == d["unit"]
    assert e["h2d_bytes_per_step"] == 0 and e["d2h_bytes_per_step"] == 0
