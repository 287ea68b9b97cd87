"""The N > 1 path of bench.py on CPU: replicas, one process per GPU, with no
data exchange, so what the ranks share is the timing protocol: the slowest
rank's time bounds the timed region and the whole-job value counts every
rank's work. Ranks here are gloo processes (world size 2, 127.0.0.1); the
reference arm is also run under torchrun, where rank 0 alone works and
prints one line."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, times, out_dir):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = bench.max_over_ranks(times[rank], world)
        dist.barrier()
        value = bench.job_value(1e9, 10, world, ms, 1e-9)
        with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
            json.dump({"ms": ms, "value": value}, f)
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_value_gloo(tmp_path):
    import torch.multiprocessing as mp
    world, times = 2, [3.0, 5.0]
    mp.start_processes(_rank_main, args=(world, _free_port(), times, str(tmp_path)), nprocs=world,
                       join=True, start_method="spawn")
    got = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    for g in got:
        assert g["ms"] == 5.0  # every rank sees the slowest rank's time
        # 2 ranks x 10 steps x 1 GB in 5 ms = 4000 GB/s for the whole job
        assert g["value"] == pytest.approx(4000.0)


def test_single_process_is_the_identity():
    assert bench.max_over_ranks(2.5, 1) == 2.5
    assert bench.job_value(2e9, 4, 1, 8.0, 1e-9) == pytest.approx(1000.0)


def test_reference_arm_under_torchrun_prints_one_line():
    env = dict(os.environ, OMP_NUM_THREADS="2")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "3",
           "--workload", "tiny_gemv_m1_k512_n256"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, env=env, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["unit"] == "GB/s"
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"
    # every key of the bench line, with the reference arm's own values
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
              "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["n_gpus"] == 2 and d["steps"] == 1 and d["warmup"] == 3 and d["higher_is_better"] is True
    assert d["config"]["workload"] == "tiny_gemv_m1_k512_n256" and d["ms_per_step"] > 0
    assert d["e2e"]["value"] == d["value"] and d["e2e"]["unit"] == d["unit"]
    assert d["e2e"]["d2h_bytes_per_step"] == 0
    cb = d["cpu_baseline"]
    assert cb["value"] == d["value"] and cb["cores"] >= 1 and cb["sample"]
