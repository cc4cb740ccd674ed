"""The N>1 host path on CPU: two gloo ranks (no GPU).

bench.py runs one replica per GPU: ranks join a process group, time their own
steps, take the maximum time and the summed work over ranks, and only rank 0
prints.  These tests run those helpers, and the reference arm, as two real
processes over gloo on 127.0.0.1."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out_dir: str):
    os.environ.update({"RANK": str(rank), "LOCAL_RANK": str(rank), "WORLD_SIZE": str(world),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    r, w, local = bench.dist_init(None)
    bench.barrier(w)
    mx = bench.max_over_ranks(1.5 + r, w)          # per-rank step time: the job takes the slowest
    sm = bench.sum_over_ranks(10.0 * (r + 1), w)    # per-rank work: the job sums it
    with open(os.path.join(out_dir, f"rank{r}.json"), "w") as f:
        json.dump({"rank": r, "world": w, "local": local, "max": mx, "sum": sm,
                   "backend": dist.get_backend()}, f)
    bench.barrier(w)
    dist.destroy_process_group()


def test_rank_helpers_over_gloo(tmp_path):
    world = 2
    mp.spawn(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    for r, d in enumerate(res):
        assert d["rank"] == r and d["world"] == world and d["local"] == r
        assert d["backend"] == "gloo"
        assert d["max"] == 2.5          # max over ranks of 1.5 + rank
        assert d["sum"] == 30.0         # 10 + 20


def test_reference_arm_two_ranks_prints_once():
    # torchrun launch as the driver does for N > 1; rank 1 exits without work
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl", "reference",
           "--gpus", "2", "--steps", "1", "--warmup", "0", "--cpu-seconds", "1"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600,
                       env={**os.environ, "OMP_NUM_THREADS": "2"})
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2
    assert d["value"] > 0 and d["unit"] == "TFLOP/s"
    assert d["cpu_baseline"]["kind"] == "oracle"
