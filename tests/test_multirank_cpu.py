"""The multi-rank path of the benchmark without a GPU: two gloo ranks on the CPU.

Each rank is one replica with its own problem (weak scaling, no data-path collective). Checked:
the job's step time is the slowest rank's (max over ranks), the job's throughput counts every
rank's bytes, the ranks meet at a barrier, and in the reference arm rank 0 alone runs the
oracle while the other rank returns without work.
"""
import argparse
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import torch
    import torch.distributed as dist
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    r, w, _ = bench._dist()
    step_ms = 10.0 + 5.0 * rank                       # rank 1 is the slow one
    job_ms = bench._max_over_ranks(step_ms, w)
    gbs = bench._job_gbs(1_000_000_000, job_ms, w)
    dist.barrier()
    args = argparse.Namespace(config=1, steps=1, warmup=0, gpus=world)
    ref = bench.run_reference(args)
    dist.barrier()
    dist.destroy_process_group()
    out.put((r, w, job_ms, gbs, None if ref is None else (ref["impl"], ref["n_gpus"], ref["value"] > 0)))


def test_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=240) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, w0, t0, g0, ref0), (r1, w1, t1, g1, ref1) = res
    assert (r0, r1) == (0, 1) and w0 == w1 == 2
    assert t0 == t1 == 15.0                            # the slowest rank's step
    assert g0 == g1 == pytest.approx(2 * 1e9 / 15e-3 / 1e9)
    assert ref0 == ("reference", 2, True) and ref1 is None
