"""The N > 1 launch path on CPU, with gloo and world size 2.

The hyper-connection path shards by tokens with no data-path collective
(replicas only): every rank runs its own batch, and the job's time is the
slowest rank's.  These tests cover that host logic without a GPU: the
max-over-ranks reduction and the per-rank seeds, in two spawned processes,
and the real torchrun launch of bench.py's reference arm on two ranks (rank 0
prints the one JSON line; rank 1 exits 0 without work)."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        got = bench.max_over_ranks(10.0 * (rank + 1))
        seed = bench.rank_seed(4, rank)
        env = bench.dist_env()
        with open(os.path.join(out_dir, "rank%d.json" % rank), "w") as fh:
            json.dump({"max": got, "seed": seed, "env": env}, fh)
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_seeds_gloo_world2(tmp_path):
    world = 2
    mp.start_processes(_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True,
                       start_method="spawn")
    res = [json.load(open(tmp_path / ("rank%d.json" % r))) for r in range(world)]
    # every rank sees the slowest rank's time
    assert [r["max"] for r in res] == [20.0, 20.0]
    # rank 0 runs the workload's own seed; the replicas draw different batches
    assert res[0]["seed"] == 4 and res[1]["seed"] == 1004
    assert [tuple(r["env"]) for r in res] == [(0, 0, 2), (1, 1, 2)]


def test_max_over_ranks_single_process_is_identity():
    import bench
    assert not dist.is_initialized()
    assert bench.max_over_ranks(3.5) == 3.5


def test_reference_arm_under_torchrun_two_ranks():
    """`bench.py --impl reference` launched the way the N > 1 bench is: one
    JSON line from rank 0, exit status 0 on every rank."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes", "1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2", "--steps", "1",
           "--warmup", "0", "--reference-tokens", "1"]
    env = dict(os.environ, OMP_NUM_THREADS="1")
    p = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600, env=env)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [ln for ln in p.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, p.stdout[-2000:]
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["n_gpus"] == 2 and rec["value"] > 0
    assert rec["cpu_baseline"]["kind"] == "oracle"
    assert rec["e2e"]["h2d_bytes_per_step"] == 0
