"""The multi-process paths of bench.py on CPU with gloo, world size 2.

With N GPUs bench.py runs one independent replica of the workload per rank (the
simulated data-parallel ranks live inside one GPU, so GPUs exchange nothing but
the timing): it times with a barrier on both sides and takes the maximum over
ranks.  The reference arm runs on rank 0 only.
"""

import json
import os
import socket
import subprocess
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # each rank's elapsed time differs; every rank must see the slowest one
        got = bench.max_over_ranks(dist, 10.0 + 5.0 * rank, "cpu")
        # a rank that cannot take part makes every rank skip the collective-bearing section
        agree = (bench.all_ranks_ok(dist, True, "cpu"), bench.all_ranks_ok(dist, rank == 0, "cpu"))
        dist.barrier()
        out[rank] = (got, agree)
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_world_size_2():
    port = _free_port()
    manager = mp.get_context("spawn").Manager()
    out = manager.dict()
    mp.start_processes(_worker, args=(2, port, out), nprocs=2, join=True, start_method="spawn")
    assert dict(out) == {0: (15.0, (True, False)), 1: (15.0, (True, False))}


def test_reference_arm_under_torchrun_prints_once():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "2", "--warmup", "1"]
    res = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [ln for ln in res.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["n_gpus"] == 2 and rec["steps"] == 2
    assert rec["value"] > 0 and rec["cpu_baseline"]["kind"] == "oracle"
    assert rec["e2e"]["h2d_bytes_per_step"] == 0


@pytest.mark.parametrize("workload", ["llama-1.3b-zero2", "gpt2-small-zero1"])
def test_reference_arm_single_process(workload):
    res = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                          "--warmup", "0", "--workload", workload], capture_output=True, text=True, timeout=600,
                         cwd=ROOT)
    assert res.returncode == 0, res.stderr[-2000:]
    rec = json.loads([ln for ln in res.stdout.splitlines() if ln.startswith("{")][0])
    assert rec["metric"].startswith("sharded AdamW step") and rec["unit"] == "params/s"
    assert rec["config"]["workload"] == workload
