"""The multi-process path of bench.py on CPU (gloo, world size 2).

The hot path shards by (batch, head) with no exchange, so N GPUs run N
independent replicas; what the ranks share is host logic: the process group
set-up, the barrier around the timed region, the max over ranks of the step
time, and the rule that rank 0 alone prints the result line.
"""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, port: int, out_dir: str):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE="2", RANK=str(rank),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import importlib.util
    spec = importlib.util.spec_from_file_location("bench", os.path.join(ROOT, "bench.py"))
    bench = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(bench)
    ws, r, local = bench.dist_setup()
    bench.dist_barrier(ws)
    # each rank's "step time"; the job's time is the slowest rank's
    worst = bench.dist_max(10.0 + 5.0 * r, ws)
    bench.dist_barrier(ws)
    with open(os.path.join(out_dir, f"rank{r}.json"), "w") as f:
        json.dump({"ws": ws, "rank": r, "local": local, "max": worst}, f)
    import torch.distributed as dist
    dist.destroy_process_group()


@pytest.mark.timeout(180)
def test_dist_max_and_barrier_over_two_gloo_ranks(tmp_path):
    import torch.multiprocessing as mp
    port = _free_port()
    mp.start_processes(_rank_main, args=(port, str(tmp_path)), nprocs=2, join=True, start_method="spawn")
    got = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(2)]
    assert [g["rank"] for g in got] == [0, 1]
    assert all(g["ws"] == 2 for g in got)
    assert all(g["max"] == 15.0 for g in got)   # both ranks see the slowest rank's time


@pytest.mark.timeout(300)
def test_reference_arm_under_torchrun_prints_one_line(tmp_path):
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--workload", "tiny", "--steps", "1", "--warmup", "1"]
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="", OMP_NUM_THREADS="2")
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=280)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    assert line["value"] > 0 and line["cpu_baseline"]["kind"] == "oracle"
    assert line["cpu_baseline"]["cores"] == 2        # the threads the oracle actually ran on
    assert line["e2e"]["h2d_bytes_per_step"] == 0
