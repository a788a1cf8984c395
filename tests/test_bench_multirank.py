"""CPU (gloo, world size 2) test of bench.py's multi-rank host logic: each rank
gets its own problem, the timing is the maximum over ranks, and the reported
value is the whole job's throughput."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from fp8_bit_attention_gb300 import workloads as W


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w = bench.rank_workload(W.WORKLOADS["small"], rank)
        my_ms = 100.0 + 50.0 * rank                    # rank 1 is the slow one
        slowest = bench.max_over_ranks(my_ms, dist, torch.device("cpu"))
        value = bench.whole_job_tflops(1e12, world, 4, slowest * 4)
        out[rank] = (w.seed, slowest, value)
    finally:
        dist.destroy_process_group()


def test_two_ranks_gloo():
    world = 2
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, _free_port(), out), nprocs=world, join=True)
        res = dict(out)
    seeds = {r: res[r][0] for r in range(world)}
    assert seeds[0] == W.WORKLOADS["small"].seed and seeds[1] != seeds[0]
    assert res[0][1] == res[1][1] == 150.0               # max over ranks, seen by both
    # 2 ranks x 1e12 flop per step, 4 steps in 600 ms -> 13.33 TFLOP/s
    assert res[0][2] == pytest.approx(2 * 1e12 * 4 / 0.6 / 1e12)


def test_single_process_defaults():
    w = W.WORKLOADS["small"]
    assert bench.rank_workload(w, 0) is w
    assert bench.max_over_ranks(3.5) == 3.5


def _bench(args, extra_env=None, timeout=180):
    import json
    import subprocess
    import sys
    env = {k: v for k, v in os.environ.items()
           if k not in ("WORLD_SIZE", "RANK", "LOCAL_RANK", "MASTER_ADDR", "MASTER_PORT")}
    env.update(extra_env or {})
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), *args], capture_output=True, text=True,
                       timeout=timeout, env=env, cwd=root)
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    return r.returncode, [json.loads(ln) for ln in lines], r.stderr


def test_gpus_flag_starts_one_rank_per_gpu():
    """`bench.py --gpus 2` run directly starts two ranks itself (through
    torch.distributed.run); both join the process group and one line reports
    n_gpus = 2."""
    rc, lines, err = _bench(["--gpus", "2", "--dry-run"])
    assert rc == 0, err
    assert len(lines) == 1
    assert lines[0]["n_gpus"] == 2 and lines[0]["ranks_joined"] == 2 and lines[0]["dry_run"] is True


def test_gpus_flag_must_match_world_size():
    rc, lines, err = _bench(["--gpus", "2", "--dry-run"],
                            {"WORLD_SIZE": "3", "RANK": "0", "LOCAL_RANK": "0"})
    assert rc != 0 and not lines
    assert "WORLD_SIZE=3" in err
    rc, lines, _ = _bench(["--dry-run"])
    assert rc == 0 and lines[0]["n_gpus"] == 1


def test_reference_arm_prints_its_line():
    """--impl reference times the CPU oracle on a bounded sample and prints
    one JSON line with the main arm's metric, its own cpu_baseline and an
    e2e entry with no host<->device bytes."""
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = {k: v for k, v in os.environ.items() if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK")}
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference", "--workload", "small",
                        "--steps", "1", "--warmup", "0"], capture_output=True, text=True, timeout=600, env=env,
                       cwd=root)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["metric"] == bench.METRIC
    assert line["value"] > 0 and line["unit"] == "TFLOP/s" and line["higher_is_better"] is True
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
    assert line["config"]["workload"] == "small"
