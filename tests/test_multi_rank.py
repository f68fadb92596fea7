"""The N > 1 path of bench.py on CPU: two ranks over gloo (no GPU).

The hot path shards by sequence with no exchange (every rank is an independent replica with its
own pool and inputs), so the only cross-rank steps are the host-side ones: each rank's inputs
come from its own seeds, the timed region is bracketed by barriers, the whole-job value is all
ranks' bytes over the slowest rank's time (a MAX all-reduce), and only rank 0 prints (the
reference arm included). These run here as two processes on 127.0.0.1.
"""
import json
import os
import socket
import subprocess
import sys
from pathlib import Path

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = Path(__file__).resolve().parents[1]
sys.path.insert(0, str(ROOT))
import bench  # noqa: E402
import workloads as W  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ws, r, local = bench.dist_env()
    assert (ws, r, local) == (world, rank, rank)
    # each rank's replica: its own seeds, so its own data
    c = W.make("tiny", seed=bench.rank_seed(W.CONFIGS["tiny"].seed, rank, 0))
    nbytes = bench.kv_bytes(c.context_lens, c.Hkv, c.D)
    elapsed = 10.0 + 5.0 * rank  # ms: rank 1 is the slower one
    dist.barrier()
    slow = bench.slowest(torch, elapsed, dist, torch.device("cpu"))
    value = bench.weak_gbs(ws, nbytes, slow)
    np.save(Path(out_dir) / f"q{rank}.npy", c.q)
    (Path(out_dir) / f"r{rank}.json").write_text(json.dumps({"slow": slow, "value": value,
                                                             "nbytes": nbytes}))
    dist.destroy_process_group()


def test_two_ranks_aggregate_over_gloo(tmp_path):
    world = 2
    mp.spawn(_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    res = [json.loads((tmp_path / f"r{r}.json").read_text()) for r in range(world)]
    # both ranks agree on the slowest time and on the whole-job value
    assert res[0]["slow"] == res[1]["slow"] == 15.0
    assert res[0]["value"] == res[1]["value"]
    assert res[0]["value"] == pytest.approx(world * res[0]["nbytes"] / 15e-3 / 1e9)
    # the replicas run on different data
    q0, q1 = np.load(tmp_path / "q0.npy"), np.load(tmp_path / "q1.npy")
    assert q0.shape == q1.shape and not np.array_equal(q0, q1)


def test_single_rank_needs_no_collective():
    assert bench.slowest(torch, 3.5, None, torch.device("cpu")) == 3.5
    assert bench.weak_gbs(1, 2e9, 1000.0) == pytest.approx(2.0)


def test_reference_arm_under_torchrun_prints_once():
    """`bench.py --impl reference` on two ranks: rank 0 alone times the oracle and prints one
    JSON line; the other rank exits 0 without work."""
    env = dict(os.environ, PYTHONPATH=str(ROOT))
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), str(ROOT / "bench.py"),
           "--impl", "reference", "--workload", "tiny", "--gpus", "2", "--steps", "3",
           "--warmup", "3"]
    r = subprocess.run(cmd, capture_output=True, text=True, cwd=ROOT, env=env, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
