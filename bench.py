#!/usr/bin/env python
"""Benchmark of the GatedDeltaNet mixer hot path on one GB300 (or N, weakly scaled).

Default workload: single-sequence chunked prefill, T=8192 tokens, 16 q/k heads,
32 v heads, dk=dv=128, chunk 64, bf16 inputs, zero initial state.  One step is
one pass of the prefill path over that batch: gate prep, causal conv1d+SiLU
(+history update), the chunked gated delta rule with in-kernel q/k L2 norm and
state out, and the gated RMSNorm.  The decode path (64 sequences x 256
one-token steps, fused conv/L2/gates/state update/norm) is measured in the same
run and reported under "decode".

Prints ONE JSON line (rank 0).  --impl reference times the fp64 CPU oracle
on a bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from gateddeltanet_linear_attention_gb300.inputs import WORKLOADS, make_inputs  # noqa: E402

METRIC = "GDN prefill tokens/s (% bf16 TC peak); decode state-update GB/s (% HBM peak)"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_FLUSH_BYTES = 512 << 20


# ------------------------------------------------------------------ helpers

def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def chunk_flops(lens, C, dk, dv, HV):
    """Algorithmic contraction FLOPs of the chunked rule: per chunk of L tokens
    and v-head, 2L^2dk (KK^T) + 2L^2dk (QK^T) + 2L^2dk (W) + 2L^2dv (U)
    + 2L^2dv (intra O) + 3*2L*dk*dv (W M, Q M, K~^T U') + 2L^3/3 (solve)."""
    tot = 0.0
    for L in lens:
        full, rem = divmod(int(L), C)
        for Lc in [C] * full + ([rem] if rem else []):
            tot += (6 * Lc * Lc * dk + 4 * Lc * Lc * dv + 6 * Lc * dk * dv + 2 * Lc ** 3 / 3)
    return tot * HV


def step_hbm_bytes(wl, T, N):
    """Algorithmic HBM bytes of one mixer prefill step: per token x (CH activations), z and y
    (HV*dv activations each) and g, beta (HV fp32 each); per sequence the fp32 state read and
    written (zero initial state: written only) and the conv history read and written."""
    a = 2 if wl.act == "bf16" else 4
    per_tok = wl.CH * a + 2 * wl.HV * wl.dv * a + 2 * wl.HV * 4
    state = wl.HV * wl.dk * wl.dv * 4 * (2 if wl.init_state else 1)
    conv = wl.CH * 3 * a * (2 if wl.init_conv else 1)
    return T * per_tok + N * (state + conv)


def src_sha(paths):
    h = hashlib.sha256()
    for p in paths:
        h.update(open(os.path.join(ROOT, p), "rb").read())
    return h.hexdigest()[:16]


def traffic_for(name):
    """DRAM bytes per launch from a committed ncu summary, if the kernel source
    has not changed since the counters were taken (else None)."""
    p = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(p):
        return None
    try:
        d = json.load(open(p)).get(name)
        if d and d.get("src_sha") == src_sha(d["sources"]):
            return d["dram_bytes_per_launch"]
    except Exception:
        return None
    return None


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""
    Q = ("index,uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid):
        self.uuid = uuid
        self.proc = None
        self.path = "/tmp/gdn_clocks_%d.csv" % os.getpid()

    def __enter__(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "--query-gpu=" + self.Q,
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if not self.proc or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 10 or (self.uuid and f[1] != self.uuid):
                continue
            try:
                sm.append(float(f[2]))
                mx = float(f[3])
            except ValueError:
                continue
            for nm, v in zip(names, f[6:10]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_init():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    if ws <= 1:
        return 0, 1, 0
    import torch.distributed as dist
    rank = int(os.environ["RANK"])
    local = int(os.environ.get("LOCAL_RANK", rank))
    backend = "nccl" if torch.cuda.is_available() else "gloo"
    if torch.cuda.is_available():
        torch.cuda.set_device(local)
    dist.init_process_group(backend)
    return rank, ws, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, ws):
    if ws == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64,
                     device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def workload_desc(wl, inp):
    lens = inp["seqlens"]
    return ("%s: N=%d, T=%d, HK=%d, HV=%d, dk=dv=%d, chunk %d, %s inputs, %s initial state"
            % (wl.name, len(lens), sum(lens), wl.HK, wl.HV, wl.dk, wl.chunk, wl.act,
               "nonzero" if wl.init_state else "zero"))


# ----------------------------------------------------------- CPU oracle arm

def oracle_sample(wl, inp, kheads, max_tokens=None):
    """Run the oracle on q/k heads `kheads` (and their v-heads) of the workload, each sequence
    cut to its first `max_tokens // N` tokens when max_tokens is given; returns (seconds,
    tokens of the sample, v-heads of the sample, threads used)."""
    import oracle
    oracle.build()
    G = wl.HV // wl.HK
    lens = list(inp["seqlens"])
    cu = inp["cu_seqlens"].tolist()
    keep = lens if max_tokens is None else [min(L, max(64, max_tokens // len(lens))) for L in lens]
    rows = np.concatenate([np.arange(cu[n], cu[n] + keep[n]) for n in range(len(lens))])
    cu_s = np.concatenate([[0], np.cumsum(keep)]).astype(np.int32)
    units = len(lens) * len(kheads) * G
    threads = max(1, min(os.cpu_count() or 1, units))
    pick = lambda t: None if t is None else t[rows]
    t0 = time.perf_counter()
    oracle.mixer_heads(pick(inp["x"]), inp["conv_w"], pick(inp["u"]), pick(inp["b_logit"]), inp["A_log"],
                       inp["dt_bias"], pick(inp["z"]), inp["norm_w"], cu_s, wl.HK, wl.HV, wl.dk, wl.dv,
                       kheads, state=inp["state"], conv_state=inp["conv_state"], n_threads=threads)
    dt = time.perf_counter() - t0
    return dt, int(sum(keep)), len(kheads) * G, threads


def run_reference(args, rank, ws):
    if rank != 0:
        return
    wl = WORKLOADS[args.workload]
    inp = make_inputs(wl)
    T = sum(inp["seqlens"])
    # bounded sample per step: half of the q/k heads (all cores busy) over the first 2048
    # tokens of the batch; the step time printed is the measured time of that sample
    kheads = list(range(max(1, wl.HK // 2)))
    cap = 2048
    for _ in range(args.warmup):
        oracle_sample(wl, inp, kheads, cap)
    times, th, toks, vh = [], 1, 0, 0
    for _ in range(args.steps):
        dt, toks, vh, th = oracle_sample(wl, inp, kheads, cap)
        times.append(dt)
    tot = sum(times)
    step_s = tot / len(times)
    value = toks * (vh / wl.HV) / step_s                # whole-token equivalents per second
    sample = ("per step: the first %d of %d tokens, %d of %d v-heads (q/k heads %d-%d); value = "
              "sample tokens x v-head fraction / measured step time" % (toks, T, vh, wl.HV, kheads[0], kheads[-1]))
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * step_s, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": workload_desc(wl, inp), "sample": sample},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": th, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ GPU arm

def run_ours(args, rank, ws, local):
    from gateddeltanet_linear_attention_gb300 import gdn
    assert torch.cuda.is_available(), "the GPU arm needs a CUDA device"
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    gdn.load()
    pk, pk_src = peaks()
    wl = WORKLOADS[args.workload]
    inp = make_inputs(wl)
    lens = inp["seqlens"]
    T, N = sum(lens), len(lens)
    cfg = gdn.make_config(wl.HK, wl.HV, wl.dk, wl.dv, wl.chunk, wl.act, n_slots=N)
    d = {k: v.to(dev) for k, v in inp.items() if hasattr(v, "to")}
    H = wl.HK * wl.dk
    stream = torch.cuda.current_stream()

    # buffers (caller-owned; nothing is allocated inside the timed region)
    y = torch.empty((T, wl.HV * wl.dv), dtype=torch.bfloat16, device=dev)
    state_out = torch.empty((N, wl.HV, wl.dk, wl.dv), device=dev)
    conv = (d["conv_state"].clone() if wl.init_conv
            else torch.zeros((N, wl.CH, 3), dtype=wl.torch_act, device=dev))
    state_in = d["state"] if wl.init_state else None
    wsp = torch.empty(max(gdn.gdn_workspace_size(cfg, T, N), 16), dtype=torch.uint8, device=dev)

    def step():
        # the whole mixer through the public fused entry point (a1-a7)
        gdn.gdn_mixer_prefill(cfg, d["x"], d["z"], d["u"], d["b_logit"], d["conv_w"], d["A_log"],
                              d["dt_bias"], d["norm_w"], d["cu_seqlens"], y, state_in=state_in,
                              state_out=state_out, conv_state=conv, workspace=wsp)

    tc_path = wl.act == "bf16" and wl.dk == 128 and wl.dv == 128 and wl.chunk == 64
    # conv (gates fused), conv-history update, chunk map, [T;PT] kernel, chain (norm fused);
    # SIMT: conv, history update, chunk, norm
    launches_per_step = 5 if tc_path else 4
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with Clocks(uuid) as clk:
        barrier(ws)
        torch.cuda.synchronize()
        e0.record(stream)
        for i in range(args.steps):
            step()
        e1.record(stream)
        torch.cuda.synchronize()
        barrier(ws)
    assert gdn.gdn_device_error() == 0
    elapsed = e0.elapsed_time(e1) / 1e3
    elapsed = max_over_ranks(elapsed, ws)
    value = ws * T * args.steps / elapsed

    # ---- the chunked rule alone (gdn_chunk_prefill on the conv output), for its roofline
    chunk_s = time_chunked_rule(gdn, cfg, wl, d, conv, wsp, state_in, state_out, max(3, min(args.steps, 20)))
    flops = chunk_flops(lens, wl.chunk, wl.dk, wl.dv, wl.HV)
    tc_peak = pk["bf16_tflops"]
    roof = {"kernel": CHUNK_KERNELS if tc_path else "chunk_simt_kernel", "bound": "tensor",
            "achieved": flops / chunk_s / 1e12,
            "peak": tc_peak, "unit": "TFLOP/s", "frac": flops / chunk_s / 1e12 / tc_peak,
            "traffic": traffic_for("chunk_prefill_8k"), "peak_source": pk_src + " bf16 burst",
            "kernel_ms": chunk_s * 1e3, "flops_per_launch": flops}
    # the whole step against both bounds: the step's algorithmic bytes (x, z, y, g and beta per
    # token, state in and out per sequence) at the copy peak and its contraction FLOPs at the
    # tensor peak, the larger over the measured step time
    step_s = elapsed / args.steps
    step_bytes = step_hbm_bytes(wl, T, N)
    t_tc, t_hbm = flops / (tc_peak * 1e12), step_bytes / (pk["hbm_gbs"] * 1e9)
    step_roof = {"scope": "one gdn_mixer_prefill step", "flops": flops, "bytes": step_bytes,
                 "tensor_floor_us": t_tc * 1e6, "hbm_floor_us": t_hbm * 1e6,
                 "bound": "hbm" if t_hbm >= t_tc else "tensor", "step_us": step_s * 1e6,
                 "frac": max(t_tc, t_hbm) / step_s, "tensor_frac": t_tc / step_s,
                 "peak_source": pk_src}

    # ---- the other prefill workloads: varlen packing and a 64K-token sequence
    legs = {}
    if not args.no_legs:
        del wsp
        torch.cuda.empty_cache()
        for name in ("varlen_16", "long_64k"):
            legs[name] = bench_prefill_leg(args, dev, gdn, pk, pk_src, name)
            torch.cuda.empty_cache()

    # ---- decode: 64 sequences x S one-token steps, L2 flushed between steps
    dec = None
    if args.decode_steps > 0:
        dec = bench_decode(args, dev, gdn, pk, pk_src)

    # ---- the same decode on a Q8 state, without and with the error-feedback residual
    dq8 = dq8e = None
    if args.decode_steps > 0:
        dq8 = bench_decode_q8(args, dev, gdn, pk, pk_src)
        dq8e = bench_decode_q8(args, dev, gdn, pk, pk_src, ef=True)

    # ---- slot snapshot (state + conv history) through gdn_state_copy
    snap = None
    if args.decode_steps > 0:
        snap = bench_state_copy(args, dev, gdn, pk, pk_src)

    # ---- multi-token verification round (8 tokens per sequence) through gdn_mixer_verify
    ver = None
    if args.decode_steps > 0:
        ver = bench_verify(args, dev, gdn, pk, pk_src)

    # ---- backward of the core rule (training) at the prefill shape
    bwd = None
    if args.decode_steps > 0:
        bwd = bench_backward(args, dev, gdn, pk, pk_src)

    # ---- end to end through the public fused call with pinned host buffers
    e2e = None
    if not args.no_e2e:
        e2e = bench_e2e(args, dev, gdn, cfg, wl, inp, d, N, T)

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu:
        dt, _, _, th = oracle_sample(wl, inp, list(range(wl.HK)))
        cpu = {"value": T / dt, "unit": "tokens/s", "cores": th, "kind": "oracle",
               "sample": "the whole workload (all %d v-heads, %d tokens), once" % (wl.HV, T)}

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws,
                "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": 1e3 * elapsed / args.steps, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None,
                "dtype": "bf16x3/fp32" if tc_path else "fp32", "data": "synthetic",
                "config": {"workload": workload_desc(wl, inp), "parallelism": "dp%d" % ws,
                           "l2": "inputs larger than L2 (x %d MiB + z %d MiB per step)"
                                 % (T * wl.CH * 2 >> 20, T * wl.HV * wl.dv * 2 >> 20),
                           "activations": wl.act, "y_dtype": "bf16"},
                "roofline": roof, "step_roofline": step_roof, "cpu_baseline": cpu, "e2e": e2e,
                "gpu_launches": launches_per_step * args.steps,
                "clocks": clk.summary(), "varlen_16": legs.get("varlen_16"), "long_64k": legs.get("long_64k"),
                "decode": dec, "decode_q8": dq8, "decode_q8_ef": dq8e, "state_copy": snap,
                "verify": ver, "backward": bwd}
        print(json.dumps(line), flush=True)


CHUNK_KERNELS = ("chunked rule: chunk_map + chunk_tp_kernel + chunk_chain_kernel (tcgen05, bf16x3 "
                 "operands), timed together through gdn_chunk_prefill")


def time_chunked_rule(gdn, cfg, wl, d, conv, wsp, state_in, state_out, reps):
    """Seconds per gdn_chunk_prefill launch on the workload's conv output (CUDA events around
    each launch, L2 evicted by a read before each, 2 untimed warm-ups)."""
    dev = d["x"].device
    T = d["x"].shape[0]
    H = wl.HK * wl.dk
    stream = torch.cuda.current_stream()
    g = torch.empty((T, wl.HV), device=dev)
    beta = torch.empty_like(g)
    xa = torch.empty((T, wl.CH), device=dev)
    o = torch.empty((T, wl.HV * wl.dv), device=dev)
    gdn.gdn_gate_prep(cfg, d["u"], d["b_logit"], d["A_log"], d["dt_bias"], g, beta)
    gdn.gdn_conv1d_prefill(cfg, d["x"], d["cu_seqlens"], d["conv_w"], conv.clone(), None, xa)
    flush = torch.empty(L2_FLUSH_BYTES // 4, device=dev)
    flush.fill_(1.0)
    sink = torch.empty((), device=dev)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(reps + 2)]
    for i in range(reps + 2):
        torch.sum(flush, 0, out=sink)
        ev[i][0].record(stream)
        gdn.gdn_chunk_prefill(cfg, xa[:, :H], xa[:, H:2 * H], xa[:, 2 * H:], g, beta,
                              d["cu_seqlens"], state_in, state_out, None, o, workspace=wsp)
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    assert gdn.gdn_device_error() == 0
    return sum(a.elapsed_time(b) for a, b in ev[2:]) / 1e3 / reps


def bench_prefill_leg(args, dev, gdn, pk, pk_src, name):
    """One more prefill workload through gdn_mixer_prefill (tokens/s over a few steps, CUDA
    events, inputs larger than L2), with its chunked rule timed alone for the roofline; the
    FLOPs count every chunk at its actual length."""
    wl = WORKLOADS[name]
    inp = make_inputs(wl)
    lens = inp["seqlens"]
    T, N = sum(lens), len(lens)
    cfg = gdn.make_config(wl.HK, wl.HV, wl.dk, wl.dv, wl.chunk, wl.act, n_slots=N)
    d = {k: v.to(dev) for k, v in inp.items() if hasattr(v, "to") and not k.startswith("dec_")}
    y = torch.empty((T, wl.HV * wl.dv), dtype=torch.bfloat16, device=dev)
    state_in = d["state"] if wl.init_state else None
    state_out = torch.empty((N, wl.HV, wl.dk, wl.dv), device=dev)
    conv0 = (d["conv_state"].clone() if wl.init_conv
             else torch.zeros((N, wl.CH, 3), dtype=wl.torch_act, device=dev))
    conv = conv0.clone()
    wsp = torch.empty(gdn.gdn_workspace_size(cfg, T, N), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def step():
        gdn.gdn_mixer_prefill(cfg, d["x"], d["z"], d["u"], d["b_logit"], d["conv_w"], d["A_log"],
                              d["dt_bias"], d["norm_w"], d["cu_seqlens"], y, state_in=state_in,
                              state_out=state_out, conv_state=conv, workspace=wsp)

    steps = 5 if T < 50000 else 3
    for _ in range(3):
        step()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    assert gdn.gdn_device_error() == 0
    step_s = e0.elapsed_time(e1) / 1e3 / steps
    chunk_s = time_chunked_rule(gdn, cfg, wl, d, conv0, wsp, state_in, state_out, 3)
    flops = chunk_flops(lens, wl.chunk, wl.dk, wl.dv, wl.HV)
    tc_peak = pk["bf16_tflops"]
    return {"workload": workload_desc(wl, inp), "value": T / step_s, "unit": "tokens/s",
            "ms_per_step": step_s * 1e3, "steps": steps, "warmup": 3,
            "roofline": {"kernel": CHUNK_KERNELS, "bound": "tensor", "achieved": flops / chunk_s / 1e12,
                         "peak": tc_peak, "unit": "TFLOP/s", "frac": flops / chunk_s / 1e12 / tc_peak,
                         "traffic": None, "peak_source": pk_src + " bf16 burst",
                         "kernel_ms": chunk_s * 1e3, "flops_per_launch": flops},
            "gpu_launches": 5 * steps}


def bench_decode(args, dev, gdn, pk, pk_src):
    wl = WORKLOADS["decode_64x256"]
    S = args.decode_steps
    from dataclasses import replace
    wl = replace(wl, decode_steps=S)
    inp = make_inputs(wl)
    N = wl.n_decode
    cfg = gdn.make_config(wl.HK, wl.HV, wl.dk, wl.dv, wl.chunk, wl.act, n_slots=N)
    state = inp["state"].to(dev)
    conv = inp["conv_state"].to(dev)
    cw, A, dt, nw = (inp[k].to(dev) for k in ("conv_w", "A_log", "dt_bias", "norm_w"))
    xs, zs, us, bs = (inp[k].to(dev) for k in ("dec_x", "dec_z", "dec_u", "dec_b_logit"))
    y = torch.empty((N, wl.HV * wl.dv), dtype=torch.bfloat16, device=dev)
    ws = torch.empty(gdn.gdn_workspace_size(cfg, N, N), dtype=torch.uint8, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, device=dev)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(S)]
    stream = torch.cuda.current_stream()
    for t in range(min(3, S)):   # warm-up on copies of the state (steps replayed below)
        st2, cv2 = state.clone(), conv.clone()
        gdn.gdn_mixer_decode(cfg, xs[t], zs[t], us[t], bs[t], cw, A, dt, nw, y, st2, cv2, ws)
    torch.cuda.synchronize()
    flush.fill_(1.0)
    torch.cuda.synchronize()
    sink = torch.empty((), device=dev)
    for t in range(S):
        # evict L2 with a read-only pass (a write flush would leave dirty lines whose
        # write-back the timed kernel would pay for)
        torch.sum(flush, 0, out=sink)
        evs[t][0].record(stream)
        gdn.gdn_mixer_decode(cfg, xs[t], zs[t], us[t], bs[t], cw, A, dt, nw, y, state, conv, ws)
        evs[t][1].record(stream)
    torch.cuda.synchronize()
    assert gdn.gdn_device_error() == 0
    ms = [a.elapsed_time(b) for a, b in evs]
    per = sum(ms) / S / 1e3
    state_bytes = 2 * N * wl.HV * wl.dk * wl.dv * 4
    gbs = state_bytes / per / 1e9
    return {"workload": "decode_64x256: 64 sequences x %d one-token steps, HK=16, HV=32, "
                        "dk=dv=128, bf16 inputs, fp32 state (128 MiB), L2 evicted by a 512 MiB read between steps"
                        % S,
            "value": gbs, "unit": "GB/s", "us_per_step": per * 1e6,
            "state_bytes_per_step": state_bytes,
            "roofline": {"kernel": "decode_prep_kernel + decode_stream_kernel (bulk-copy ring)", "bound": "hbm",
                         "achieved": gbs,
                         "peak": pk["hbm_gbs"], "unit": "GB/s", "frac": gbs / pk["hbm_gbs"],
                         "traffic": traffic_for("decode_64x256"),
                         "peak_source": pk_src + " copy"},
            "gpu_launches": 2 * S}


def bench_decode_q8(args, dev, gdn, pk, pk_src, ef=False):
    """decode_64x256 on a Q8 state pool (int8 codes + fp32 row scales, and with ef the bf16
    error-feedback residual) through gdn_mixer_decode_q8, L2 evicted between steps like the
    fp32 decode."""
    wl = WORKLOADS["decode_64x256"]
    S = args.decode_steps
    from dataclasses import replace
    wl = replace(wl, decode_steps=S)
    inp = make_inputs(wl)
    N = wl.n_decode
    cfg = gdn.make_config(wl.HK, wl.HV, wl.dk, wl.dv, wl.chunk, wl.act, n_slots=N)
    codes = torch.empty((N, wl.HV, wl.dk, wl.dv), dtype=torch.int8, device=dev)
    scales = torch.empty((N, wl.HV, wl.dk), device=dev)
    res = (torch.empty((N, wl.HV, wl.dk, wl.dv), dtype=torch.bfloat16, device=dev) if ef else None)
    gdn.gdn_state_to_q8(cfg, inp["state"].to(dev), codes, scales, 0, residual=res)
    conv = inp["conv_state"].to(dev)
    cw, A, dt, nw = (inp[k].to(dev) for k in ("conv_w", "A_log", "dt_bias", "norm_w"))
    xs, zs, us, bs = (inp[k].to(dev) for k in ("dec_x", "dec_z", "dec_u", "dec_b_logit"))
    y = torch.empty((N, wl.HV * wl.dv), dtype=torch.bfloat16, device=dev)
    ws = torch.empty(gdn.gdn_workspace_size(cfg, N, N), dtype=torch.uint8, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, device=dev)
    flush.fill_(1.0)
    sink = torch.empty((), device=dev)
    stream = torch.cuda.current_stream()
    for t in range(min(3, S)):   # warm-up on copies of the pool
        c2, s2, v2 = codes.clone(), scales.clone(), conv.clone()
        r2 = None if res is None else res.clone()
        gdn.gdn_mixer_decode_q8(cfg, xs[t], zs[t], us[t], bs[t], cw, A, dt, nw, y, c2, s2, v2, 1 + t, ws,
                                residual=r2)
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(S)]
    for t in range(S):
        torch.sum(flush, 0, out=sink)
        evs[t][0].record(stream)
        gdn.gdn_mixer_decode_q8(cfg, xs[t], zs[t], us[t], bs[t], cw, A, dt, nw, y, codes, scales, conv,
                                1 + t, ws, residual=res)
        evs[t][1].record(stream)
    torch.cuda.synchronize()
    assert gdn.gdn_device_error() == 0
    per = sum(a.elapsed_time(b) for a, b in evs) / S / 1e3
    q8_bytes = 2 * N * wl.HV * (wl.dk * wl.dv * (3 if ef else 1) + wl.dk * 4)
    gbs = q8_bytes / per / 1e9
    what = ("int8 codes + fp32 row scales + bf16 error-feedback residual, 48.5 KiB per head" if ef
            else "int8 codes + fp32 row scales, 16.5 KiB per head")
    return {"workload": "decode_64x256 with a Q8 state (%s), %d steps, L2 evicted between steps" % (what, S),
            "value": gbs, "unit": "GB/s", "us_per_step": per * 1e6, "state_bytes_per_step": q8_bytes,
            "roofline": {"kernel": "decode_prep_kernel + decode_stream_kernel (Q8 slots)", "bound": "hbm",
                         "achieved": gbs, "peak": pk["hbm_gbs"], "unit": "GB/s",
                         "frac": gbs / pk["hbm_gbs"],
                         "traffic": None if ef else traffic_for("decode_64x256_q8"),
                         "peak_source": pk_src + " copy"},
            "gpu_launches": 2 * S}


def bench_state_copy(args, dev, gdn, pk, pk_src):
    """Snapshot of the decode workload's 64 live slots (fp32 state + bf16 conv history) into 64
    snapshot rows of the same pool, through gdn_state_copy; L2 evicted before each launch."""
    wl = WORKLOADS["decode_64x256"]
    N = wl.n_decode
    cfg = gdn.make_config(wl.HK, wl.HV, wl.dk, wl.dv, wl.chunk, wl.act, n_slots=2 * N)
    state = torch.zeros((2 * N, wl.HV, wl.dk, wl.dv), device=dev)
    conv = torch.zeros((2 * N, wl.CH, 3), dtype=wl.torch_act, device=dev)
    state[:N].normal_(0.0, 0.02)
    conv[:N].normal_()
    live = torch.arange(N, dtype=torch.int32, device=dev)
    snap = live + N
    flush = torch.empty(L2_FLUSH_BYTES // 4, device=dev)
    flush.fill_(1.0)
    sink = torch.empty((), device=dev)
    stream = torch.cuda.current_stream()
    reps = max(5, min(args.decode_steps, 20))
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(reps + 3)]
    for i in range(reps + 3):           # 3 untimed warm-ups
        torch.sum(flush, 0, out=sink)
        evs[i][0].record(stream)
        gdn.gdn_state_copy(cfg, state, conv, state, conv, live, snap)
        evs[i][1].record(stream)
    torch.cuda.synchronize()
    assert gdn.gdn_device_error() == 0
    assert torch.equal(state[:N], state[N:]) and torch.equal(conv[:N], conv[N:])
    per = sum(a.elapsed_time(b) for a, b in evs[3:]) / reps / 1e3
    moved = 2 * N * (wl.HV * wl.dk * wl.dv * 4 + wl.CH * 3 * 2)
    gbs = moved / per / 1e9
    return {"workload": "snapshot of 64 live slots (fp32 state 2 MiB + bf16 conv history 48 KiB "
                        "each) into 64 rows of the same pool, L2 evicted before each launch",
            "value": gbs, "unit": "GB/s", "us_per_launch": per * 1e6, "bytes_per_launch": moved,
            "roofline": {"kernel": "state_copy_kernel", "bound": "hbm", "achieved": gbs,
                         "peak": pk["hbm_gbs"], "unit": "GB/s", "frac": gbs / pk["hbm_gbs"],
                         "traffic": None, "peak_source": pk_src + " copy"},
            "gpu_launches": reps}


def bench_verify(args, dev, gdn, pk, pk_src, k=8):
    """One verification round of k tokens for the decode workload's 64 sequences through
    gdn_mixer_verify: each head state read once and written k times (one checkpoint column per
    token); L2 evicted before each launch."""
    wl = WORKLOADS["decode_64x256"]
    N = wl.n_decode
    slots = N + N * k
    cfg = gdn.make_config(wl.HK, wl.HV, wl.dk, wl.dv, wl.chunk, wl.act, n_slots=slots)
    g = torch.Generator(device=dev).manual_seed(7)
    rn = lambda *s: torch.randn(*s, generator=g, device=dev)
    state = torch.zeros((slots, wl.HV, wl.dk, wl.dv), device=dev)
    state[:N] = rn(N, wl.HV, wl.dk, wl.dv) * 0.02
    conv = torch.zeros((slots, wl.CH, 3), dtype=wl.torch_act, device=dev)
    conv[:N] = rn(N, wl.CH, 3).to(wl.torch_act)
    x = rn(N * k, wl.CH).to(wl.torch_act); z = rn(N * k, wl.HV * wl.dv).to(wl.torch_act)
    u = rn(N * k, wl.HV).to(wl.torch_act); b = rn(N * k, wl.HV).to(wl.torch_act)
    cw = (rn(wl.CH, 4) * 0.25).to(wl.torch_act)
    A = torch.rand(wl.HV, generator=g, device=dev) * 2 - 1
    dt = torch.zeros(wl.HV, device=dev); nw = torch.ones(wl.dv, device=dev)
    y = torch.empty((N * k, wl.HV * wl.dv), dtype=torch.bfloat16, device=dev)
    src = torch.arange(N, dtype=torch.int32, device=dev)
    ckpt = N + k * src
    ws = torch.empty(gdn.gdn_workspace_size(cfg, N * k, N), dtype=torch.uint8, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, device=dev)
    flush.fill_(1.0)
    sink = torch.empty((), device=dev)
    stream = torch.cuda.current_stream()
    reps = max(5, min(args.decode_steps, 20))
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(reps + 3)]
    for i in range(reps + 3):           # 3 untimed warm-ups
        torch.sum(flush, 0, out=sink)
        evs[i][0].record(stream)
        gdn.gdn_mixer_verify(cfg, x, z, u, b, cw, A, dt, nw, y, state, conv, ckpt, k, ws,
                             state_idx=src)
        evs[i][1].record(stream)
    torch.cuda.synchronize()
    assert gdn.gdn_device_error() == 0
    per = sum(a.elapsed_time(b) for a, b in evs[3:]) / reps / 1e3
    moved = (1 + k) * N * wl.HV * wl.dk * wl.dv * 4
    gbs = moved / per / 1e9
    return {"workload": "verification round: 64 sequences x %d tokens, HK=16, HV=32, dk=dv=128, "
                        "bf16 inputs; each 64 KiB head state read once and written to %d "
                        "checkpoint columns; L2 evicted before each launch" % (k, k),
            "value": gbs, "unit": "GB/s", "us_per_round": per * 1e6,
            "tokens_per_s": N * k / per, "state_bytes_per_round": moved,
            "roofline": {"kernel": "verify_kernel (one launch per round)", "bound": "hbm",
                         "achieved": gbs, "peak": pk["hbm_gbs"], "unit": "GB/s",
                         "frac": gbs / pk["hbm_gbs"], "traffic": traffic_for("verify_64x8"),
                         "peak_source": pk_src + " copy"},
            "gpu_launches": reps}


def bench_backward(args, dev, gdn, pk, pk_src):
    """The gated delta rule core backward on one 8,192-token sequence at the prefill shape
    (HV=32, dk=dv=128, chunk 64, nonzero initial state): gdn_chunk_states once (what the
    training forward retains: the boundary states and every token's p and w), then
    gdn_chunk_backward timed per call with CUDA events, reading the retained p and w; the form
    that recomputes them is timed beside it."""
    wl = WORKLOADS["prefill_8k"]
    T, HK, HV, d, C = 8192, wl.HK, wl.HV, wl.dk, wl.chunk
    cfg = gdn.make_config(HK, HV, d, d, C, "bf16", n_slots=1)
    g = torch.Generator(device=dev).manual_seed(11)
    rn = lambda *s: torch.randn(*s, generator=g, device=dev)
    unit = lambda x: x / x.norm(dim=-1, keepdim=True)
    q = unit(rn(T, HK, d)).reshape(T, HK * d).to(torch.bfloat16)
    k = unit(rn(T, HK, d)).reshape(T, HK * d).to(torch.bfloat16)
    v = rn(T, HV * d).to(torch.bfloat16)
    gl = -torch.nn.functional.softplus(rn(T, HV)) * 0.5
    beta = torch.sigmoid(rn(T, HV))
    S0 = rn(1, HV, d, d) * 0.02
    d_o = rn(T, HV * d); dS = rn(1, HV, d, d) * 0.1
    cu = torch.tensor([0, T], dtype=torch.int32, device=dev)
    nb = gdn.chunk_count([T], C)
    bnd = torch.empty((nb, HV, d, d), device=dev)
    pw = torch.empty((T, HV, 2, d), device=dev)
    ws = torch.empty(gdn.gdn_backward_workspace_size(cfg, T, 1), dtype=torch.uint8, device=dev)
    dq = torch.empty((T, HK * d), device=dev); dk = torch.empty_like(dq)
    dv = torch.empty((T, HV * d), device=dev); dg = torch.empty((T, HV), device=dev)
    db = torch.empty_like(dg); dS0 = torch.empty_like(S0)
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    gdn.gdn_chunk_states(cfg, k, v, gl, beta, cu, bnd, ws, state_in=S0, token_pw=pw)
    e1.record(stream)
    torch.cuda.synchronize()
    states_s = e0.elapsed_time(e1) / 1e3
    reps = 3

    def timed(token_pw):
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(reps + 1)]
        for i in range(reps + 1):           # 1 untimed warm-up
            evs[i][0].record(stream)
            gdn.gdn_chunk_backward(cfg, q, k, v, gl, beta, cu, bnd, d_o, dq, dk, dv, dg, db, ws,
                                   d_state_out=dS, d_state_in=dS0, token_pw=token_pw)
            evs[i][1].record(stream)
        torch.cuda.synchronize()
        assert gdn.gdn_device_error() == 0
        return sum(a.elapsed_time(b) for a, b in evs[1:]) / reps / 1e3

    per_recompute = timed(None)
    per = timed(pw)
    # bytes the token-level algorithm moves: per pair of tokens and v-head the state before the
    # even token written to and read back from the chunk scratch, plus the boundary state per
    # chunk and the retained p and w per token
    moved = T * HV * d * d * 4 + nb * HV * d * d * 4 + T * HV * 2 * d * 4
    return {"workload": "prefill_8k shape: one 8,192-token sequence, HK=16, HV=32, dk=dv=128, "
                        "chunk 64, bf16 q/k/v, nonzero initial state, d_o and d_state_out given",
            "tokens_per_s": T / per, "ms_per_call": per * 1e3, "states_ms": states_s * 1e3,
            "ms_per_call_recomputing_p_w": per_recompute * 1e3,
            "roofline": {"kernel": "bwd_gm_kernel + bwd_kernel + bwd_group_sum_kernel", "bound": "latency",
                         "bytes_per_call": moved, "achieved": moved / per / 1e9, "unit": "GB/s",
                         "peak": pk["hbm_gbs"], "frac": moved / per / 1e9 / pk["hbm_gbs"],
                         "peak_source": pk_src + " copy", "traffic": traffic_for("backward_8k"),
                         "note": "384 CTAs (v-head x 32-column state slice x three segments of the "
                                 "sequence, 3 per SM) walk about 2,731 tokens each, replaying each "
                                 "chunk from the p and w that gdn_chunk_states retained; the "
                                 "gradients entering the later segments come from a pass over them "
                                 "that needs no forward state"},
            "gpu_launches": 8 * reps}


def bench_e2e(args, dev, gdn, cfg, wl, inp, d, N, T):
    """End to end through gdn_mixer_prefill: every step copies its inputs from pinned host
    memory and reads y back, inside the timed region.  Like a serving loop, the copies of step
    i+1 (and the read-back of step i-1) run on their own streams while step i computes, with
    two device buffer sets."""
    hx = inp["x"].pin_memory(); hz = inp["z"].pin_memory()
    hu = inp["u"].pin_memory(); hb = inp["b_logit"].pin_memory()
    hy = [torch.empty((T, wl.HV * wl.dv), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    dins = [tuple(torch.empty_like(t, device=dev) for t in (hx, hz, hu, hb)) for _ in range(2)]
    ys = [torch.empty((T, wl.HV * wl.dv), dtype=torch.bfloat16, device=dev) for _ in range(2)]
    st = torch.empty((N, wl.HV, wl.dk, wl.dv), device=dev)
    conv = torch.zeros((N, wl.CH, 3), dtype=wl.torch_act, device=dev)
    ws = torch.empty(gdn.gdn_workspace_size(cfg, T, N), dtype=torch.uint8, device=dev)
    sin = d["state"] if wl.init_state else None
    main = torch.cuda.current_stream()
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev = lambda: torch.cuda.Event()
    ev_in, ev_comp, ev_out = [ev(), ev()], [ev(), ev()], [ev(), ev()]
    used = [False, False]

    def step(i):
        k = i & 1
        dx, dz, du, db = dins[k]
        with torch.cuda.stream(s_in):
            if used[k]:
                s_in.wait_event(ev_comp[k])      # step i-2 is done reading this input set
            for h, t in ((hx, dx), (hz, dz), (hu, du), (hb, db)):
                t.copy_(h, non_blocking=True)
            ev_in[k].record(s_in)
        main.wait_event(ev_in[k])
        if used[k]:
            main.wait_event(ev_out[k])           # y of step i-2 has been read back
        gdn.gdn_mixer_prefill(cfg, dx, dz, du, db, d["conv_w"], d["A_log"], d["dt_bias"],
                              d["norm_w"], d["cu_seqlens"], ys[k], state_in=sin, state_out=st,
                              conv_state=conv, workspace=ws, stream=main)
        ev_comp[k].record(main)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_comp[k])
            hy[k].copy_(ys[k], non_blocking=True)
            ev_out[k].record(s_out)
        used[k] = True

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(main)
    for i in range(args.steps):
        step(args.warmup + i)
    for k in range(2):
        main.wait_event(ev_out[k])               # the last read-backs are inside the region
    e1.record(main)
    torch.cuda.synchronize()
    el = e0.elapsed_time(e1) / 1e3
    h2d = sum(t.numel() * t.element_size() for t in (hx, hz, hu, hb))
    return {"value": T * args.steps / el, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": hy[0].numel() * hy[0].element_size(),
            "overlap": "copies of step i+1 and read-back of step i-1 overlap step i (2 buffer sets)"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="prefill_8k", choices=["prefill_8k", "varlen_16"])
    ap.add_argument("--decode-steps", type=int, default=256)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-legs", action="store_true", help="skip the varlen_16 / long_64k prefill legs")
    args = ap.parse_args()
    rank, ws, local = dist_init()
    if args.impl == "reference":
        run_reference(args, rank, ws)
    else:
        run_ours(args, rank, ws, local)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
