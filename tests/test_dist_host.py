"""The multi-process path of bench.py on CPU (gloo, world_size 2): process-group
set-up from the torchrun environment, the barrier, and the max-over-ranks
reduction of the timed region.  The mixer itself shards by sequence and head
with no data exchange, so this host logic is all the N > 1 path adds."""
import importlib.util
import os
import socket

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    b = _bench()
    r, ws, local = b.dist_init()
    assert (r, ws, local) == (rank, world, rank)
    b.barrier(ws)
    out[rank] = b.max_over_ranks(1.5 * (rank + 1), ws)     # each rank's elapsed seconds
    import torch.distributed as dist
    dist.destroy_process_group()


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_gloo_world2_barrier_and_max_over_ranks():
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert dict(out) == {0: 3.0, 1: 3.0}


def test_single_process_needs_no_process_group(monkeypatch):
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    b = _bench()
    assert b.dist_init() == (0, 1, 0)
    assert b.max_over_ranks(2.5, 1) == 2.5
