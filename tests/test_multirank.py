"""The benchmark's multi-rank host logic on CPU with gloo (world_size 2):
timings reduce to the max over ranks, and the reference arm runs on rank 0
only (the others return without work)."""
import os
import socket

import pytest
import torch.multiprocessing as mp

from conftest import ROOT


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    got = bench.max_over_ranks(10.0 + rank * 5.0)
    import argparse
    args = argparse.Namespace(ref_sample_m=16, ref_sample_n=32, warmup=0, steps=1)
    ref = bench.reference_arm(args) if rank != 0 else "skipped"
    dist.barrier()
    dist.destroy_process_group()
    q.put((rank, got, ref))


def test_two_rank_gloo_timing_reduction_and_reference_rank_split():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict((r, (g, ref)) for r, g, ref in (q.get(timeout=120) for _ in procs))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res[0][0] == 15.0 and res[1][0] == 15.0      # max over ranks on every rank
    assert res[1][1] is None                            # non-zero ranks do no reference work


def test_single_process_identity():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5) == 3.5
