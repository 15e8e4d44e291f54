"""The multi-process path on CPU (gloo, world_size 2): process-group set-up
from the torchrun environment, the barrier, and the max-over-ranks reduction
of bench.py's timed region; and the partition the N > 1 path relies on: the
mixer shards by (sequence, q/k-head group) with no data exchange, so two
ranks that each run the oracle on their half of the heads (or of the
sequences) and gather the pieces reproduce the single-process result exactly."""
import importlib.util
import os
import socket

import numpy as np
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


def _shard_worker(rank, world, port, out):
    import torch.distributed as dist
    import oracle
    from gateddeltanet_linear_attention_gb300.inputs import Workload, make_inputs
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    wl = Workload("shard", HK=4, HV=8, dk=16, dv=16, chunk=16, act="bf16", seed=71,
                  seqlens=(30, 9, 41, 20), init_state=True, init_conv=True)
    inp = make_inputs(wl)
    args = (inp["x"], inp["conv_w"], inp["u"], inp["b_logit"], inp["A_log"], inp["dt_bias"], inp["z"],
            inp["norm_w"])
    # head shard: q/k heads rank, rank + 2 (with their v-heads), all sequences
    mine = [rank, rank + 2]
    r = oracle.mixer_heads(*args, inp["cu_seqlens"], wl.HK, wl.HV, wl.dk, wl.dv, mine,
                           state=inp["state"], conv_state=inp["conv_state"], n_threads=1)
    got = [None] * world
    dist.all_gather_object(got, (mine, r["y"], r["state"], r["conv_state"]))
    # sequence shard: sequences rank, rank + 2, all heads
    cu = inp["cu_seqlens"].tolist()
    seqs = [rank, rank + 2]
    rows = np.concatenate([np.arange(cu[n], cu[n + 1]) for n in seqs])
    cu_s = np.concatenate([[0], np.cumsum([cu[n + 1] - cu[n] for n in seqs])]).astype(np.int32)
    rs = oracle.mixer(inp["x"][rows], inp["conv_w"], inp["u"][rows], inp["b_logit"][rows], inp["A_log"],
                      inp["dt_bias"], inp["z"][rows], inp["norm_w"], cu_s, wl.HK, wl.HV, wl.dk, wl.dv,
                      state=oracle._f64(inp["state"])[seqs], conv_state=oracle._f64(inp["conv_state"])[seqs],
                      n_threads=1)
    got_s = [None] * world
    dist.all_gather_object(got_s, (seqs, rows, rs["y"], rs["state"], rs["conv_state"]))
    if rank == 0:
        full = oracle.mixer(*args, inp["cu_seqlens"], wl.HK, wl.HV, wl.dk, wl.dv, state=inp["state"],
                            conv_state=inp["conv_state"], n_threads=1)
        y = np.full_like(full["y"], np.nan); st = np.full_like(full["state"], np.nan)
        cv = np.full_like(full["conv_state"], np.nan)
        for heads, yy, ss, cc in got:
            chs, vh, cols = oracle.head_channels(wl.HK, wl.HV, wl.dk, wl.dv, heads)
            y[:, cols] = yy; st[:, vh] = ss; cv[:, chs] = cc
        heads_ok = (np.array_equal(y, full["y"]) and np.array_equal(st, full["state"])
                    and np.array_equal(cv, full["conv_state"]))
        y = np.full_like(full["y"], np.nan); st = np.full_like(full["state"], np.nan)
        cv = np.full_like(full["conv_state"], np.nan)
        for sq, rw, yy, ss, cc in got_s:
            y[rw] = yy; st[sq] = ss; cv[sq] = cc
        seqs_ok = (np.array_equal(y, full["y"]) and np.array_equal(st, full["state"])
                   and np.array_equal(cv, full["conv_state"]))
        out["ok"] = (heads_ok, seqs_ok)
    dist.destroy_process_group()


def test_gloo_world2_head_and_sequence_shards_reproduce_the_full_mixer():
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    port = _free_port()
    procs = [ctx.Process(target=_shard_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=300)
        assert p.exitcode == 0
    assert out["ok"] == (True, True)
