"""The N > 1 host path of bench.py on CPU, world size 2 over gloo: process
group set-up, the max over ranks and the barrier that bracket the timed
region, the per-rank shards (replicas: each rank its own seeded batch, no
collective on the data path), and the reference arm under torchrun, which
rank 0 alone runs and prints.
"""
import json
import os
import socket
import subprocess
import sys

import numpy as np
import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, queue):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench

    r, w, _ = bench.dist_setup(None)
    top = bench.all_max(10.0 * rank + 0.5, w)  # the slowest rank's time
    bench.barrier(w)
    b = bench.make_batch("llama", "cpu", seed_offset=r, batch=3)
    queue.put((r, w, top, b.seq_lens.tolist()))
    bench.barrier(w)
    torch.distributed.destroy_process_group()


def test_max_over_ranks_barrier_and_shards_on_two_gloo_ranks():
    ctx = torch.multiprocessing.get_context("spawn")
    queue = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, queue)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(queue.get(timeout=240) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [(r, w, top) for r, w, top, _ in got] == [(0, 2, 10.5), (1, 2, 10.5)]
    # each rank decodes its own batch: weak scaling by sequence
    assert got[0][3] != got[1][3]


@pytest.mark.timeout(600)
def test_reference_arm_under_torchrun_prints_once_from_rank_0():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), "bench.py",
           "--impl", "reference", "--workload", "block_copy", "--batch", "4", "--gpus", "2",
           "--steps", "1", "--warmup", "3"]
    env = dict(os.environ, OMP_NUM_THREADS="1")
    out = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=580, env=env)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["unit"] == "GB/s"
    assert d["cpu_baseline"]["kind"] == "oracle" and np.isfinite(d["ms_per_step"])
