"""The benchmark's multi-rank logic on CPU (gloo, world size 2).

Paged decode shards by batch: each rank decodes its own batch with no
data-path collective, and the only collectives are the timing barrier and the
max / sum reductions of the timings and byte counts (weak scaling). These
tests run that host logic in two gloo processes, and check that the reference
arm prints its line on rank 0 only.
"""
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


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank: int, world: int, port: int, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    from paged_kv_cache_context_gb300 import workloads as wl
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        assert bench.rank_info() == (rank, rank, world)
        bench.barrier()
        elapsed = 0.5 + rank           # seconds each rank timed
        nbytes = 1000.0 * (rank + 1)   # bytes each rank moved
        mx = bench.all_reduce(elapsed, "max")
        tot = bench.all_reduce(nbytes, "sum")
        # each rank draws its own batch of the same shape (weak scaling)
        case = wl.config("tiny", seed=None if rank == 0 else 50_000 + rank)
        digest = float(case.query.float().sum())
        sums = [torch.zeros(1, dtype=torch.float64) for _ in range(world)]
        dist.all_gather(sums, torch.tensor([digest], dtype=torch.float64))
        q.put((rank, mx, tot, tuple(case.query.shape), [float(s) for s in sums]))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_reduce_timings_and_draw_their_own_batches():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    got.sort()
    for rank, mx, tot, shape, sums in got:
        assert mx == 1.5 and tot == 3000.0   # whole-job value = sum of bytes / max of times
        assert shape == got[0][3]
        assert sums[0] != sums[1]             # different batches on the two ranks


def test_all_reduce_is_the_identity_without_a_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert not dist.is_initialized()
    assert bench.all_reduce(2.5, "max") == 2.5 and bench.all_reduce(2.5, "sum") == 2.5
    bench.barrier()


@pytest.mark.parametrize("rank", [0, 1])
def test_reference_arm_prints_on_rank_zero_only(rank):
    env = dict(os.environ, RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE="2",
               MASTER_ADDR="127.0.0.1", MASTER_PORT=str(_free_port()), CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "tiny", "--steps", "3", "--warmup", "3", "--gpus", "2"],
                       capture_output=True, text=True, env=env, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    if rank:
        assert lines == []
        return
    line = json.loads(lines[-1])
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
    assert line["value"] > 0 and line["steps"] == 3
