"""The bench's multi-rank plumbing on the host: the path itself does not shard (each rank runs
an independent replica), so what N > 1 adds is the process group, the barrier around the timed
region and the MAX of the step times over ranks.  Two gloo ranks on the CPU exercise it, and
the reference arm under torchrun prints exactly one line (rank 0) and exits 0 on every rank."""
import json
import os
import socket
import subprocess
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE="2",
                      RANK=str(rank), LOCAL_RANK=str(rank), CUDA_VISIBLE_DEVICES="")
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist

    r, world, _ = bench.dist_init(2)
    bench.barrier(world)
    results[r] = bench.dist_max(1.5 + r, world)  # rank 1 is the slower one
    bench.barrier(world)
    dist.destroy_process_group()


def test_two_gloo_ranks_reduce_the_slowest_time():
    port = _free_port()
    with mp.Manager() as m:
        results = m.dict()
        mp.spawn(_rank_main, args=(port, results), nprocs=2, join=True)
        assert dict(results) == {0: 2.5, 1: 2.5}


def test_reference_arm_under_torchrun_prints_once():
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes", "1", "--nproc-per-node",
           "2", "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), "bench.py",
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "3",
           "--workload", "tiny_T4_E64"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [json.loads(l) for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    line = lines[0]
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["config"]["parallelism"] == "replicas"
