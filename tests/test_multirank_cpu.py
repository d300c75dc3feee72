"""The N > 1 host path of bench.py on CPU: world-size-2 gloo ranks (rendezvous on 127.0.0.1).

bench.py runs one process per GPU; with N > 1 every rank times its own replica, the ranks meet at a
barrier around the timed region and the reported time is the maximum over ranks.  These tests run that
host logic (rank/world from the environment, barrier, max-reduction) and the reference arm under
torch.distributed.run with two CPU ranks, where only rank 0 works and prints.
"""
import json
import os
import socket
import subprocess
import sys

import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_body(rank: int, world: int, port: int, result_dir: str):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    w, r, local = bench.dist_setup()
    dist.init_process_group("gloo", rank=r, world_size=w)
    try:
        bench.barrier(w)
        slowest = bench.reduce_max(10.0 * (r + 1), w)  # each rank's own time; the report takes the max
        bench.barrier(w)
        with open(os.path.join(result_dir, f"rank{r}.txt"), "w") as f:
            f.write(f"{w} {r} {local} {slowest}\n")
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_barrier_and_max_over_ranks(tmp_path):
    port = _free_port()
    mp.spawn(_rank_body, args=(2, port, str(tmp_path)), nprocs=2, join=True)
    for r in range(2):
        w, rr, local, slowest = open(tmp_path / f"rank{r}.txt").read().split()
        assert (int(w), int(rr), int(local)) == (2, r, r)
        assert float(slowest) == 20.0


def test_reference_arm_under_torchrun_two_ranks():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "1", "--context", "512",
           "--pool-rows", "1024", "--layers", "1"]
    p = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [l for l in p.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1  # rank 0 alone prints
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["n_gpus"] == 2 and rec["value"] > 0
    assert rec["cpu_baseline"]["kind"] == "oracle"
