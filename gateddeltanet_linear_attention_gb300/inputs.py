"""Seeded synthetic inputs for the GatedDeltaNet mixer.

This module draws random numbers and rounds them to the activation dtype; it
holds none of the mixer's arithmetic.  Both the CUDA path and the CPU checker
consume exactly the tensors produced here.

Distributions (the mixer workloads the library is measured and checked on):
  x (raw q|k|v projection)  ~ N(0, 1)                       [T, CH]      act dtype
  conv weights              ~ N(0, std 0.25)                [CH, 4]      act dtype
  A_log                     ~ U(-1, 1)                      [HV]         fp32
  dt_bias                   = 0                             [HV]         fp32
  u (decay projection)      ~ N(0, 1)                       [T, HV]      act dtype
  b_logit (beta projection) ~ N(0, 1)                       [T, HV]      act dtype
  z (norm gate)             ~ N(0, 1)                       [T, HV*dv]   act dtype
  norm weight               = 1                             [dv]         fp32
  initial state (if any)    ~ N(0, std 0.02)                [N, HV, dk, dv] fp32
  conv history (if any)     ~ N(0, 1)                       [N, CH, 3]   act dtype
bf16 values are drawn in fp32 and rounded once, round-to-nearest-even.
Draw order is fixed (lengths, x, conv_w, A_log, u, b_logit, z, state, conv
history, then the decode steps' x, u, b_logit, z) so a seed fixes every value.
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    HK: int
    HV: int
    dk: int
    dv: int
    chunk: int
    act: str                       # "bf16" | "fp32"
    seed: int
    seqlens: tuple = ()            # prefill lengths (empty: no prefill)
    init_state: bool = False
    init_conv: bool = False
    decode_steps: int = 0          # one-token steps after the prefill
    n_decode: int = 0              # sequences decoded per step (0: = number of prefill sequences)
    varlen: tuple = ()             # (n, lo, hi): lengths drawn from U[lo, hi] with the seed

    @property
    def CH(self) -> int:
        return 2 * self.HK * self.dk + self.HV * self.dv

    @property
    def n_seqs(self) -> int:
        if self.varlen:
            return self.varlen[0]
        return len(self.seqlens) if self.seqlens else self.n_decode

    @property
    def torch_act(self):
        return torch.bfloat16 if self.act == "bf16" else torch.float32


# The five workloads the mixer is checked and measured on.
WORKLOADS = {
    # tiny fp32 mixer: one sequence of 64 tokens, 2 heads, d=32, chunk 16, zero state
    "tiny_fp32": Workload("tiny_fp32", HK=2, HV=2, dk=32, dv=32, chunk=16, act="fp32", seed=0,
                          seqlens=(64,)),
    # recurrent decode: 64 sequences x 256 one-token steps, HK=16, HV=32, d=128
    "decode_64x256": Workload("decode_64x256", HK=16, HV=32, dk=128, dv=128, chunk=64,
                              act="bf16", seed=1, init_state=True, init_conv=True,
                              decode_steps=256, n_decode=64),
    # single-sequence chunked prefill, T=8192
    "prefill_8k": Workload("prefill_8k", HK=16, HV=32, dk=128, dv=128, chunk=64, act="bf16",
                           seed=2, seqlens=(8192,)),
    # varlen packed prefill: 16 sequences, lengths U[256, 4096], nonzero state and history
    "varlen_16": Workload("varlen_16", HK=16, HV=32, dk=128, dv=128, chunk=64, act="bf16",
                          seed=3, varlen=(16, 256, 4096), init_state=True, init_conv=True),
    # long context: 65,536-token prefill, then 512 decode steps from its state
    "long_64k": Workload("long_64k", HK=16, HV=32, dk=128, dv=128, chunk=64, act="bf16", seed=4,
                         seqlens=(65536,), decode_steps=512),
}


def shrink(wl: Workload, **kw) -> Workload:
    """A smaller variant of a workload (same dims unless overridden)."""
    return replace(wl, **kw)


def _normal(gen, shape, std=1.0):
    return torch.randn(shape, generator=gen, dtype=torch.float32) * std


def make_inputs(wl: Workload) -> dict:
    """All inputs of a workload as CPU tensors (act dtype / fp32 / int32)."""
    gen = torch.Generator().manual_seed(wl.seed)
    act = wl.torch_act
    if wl.varlen:
        n, lo, hi = wl.varlen
        lens = torch.randint(lo, hi + 1, (n,), generator=gen, dtype=torch.int64).tolist()
    else:
        lens = list(wl.seqlens)
    T = int(sum(lens))
    N = len(lens) if lens else wl.n_decode
    cu = torch.zeros(len(lens) + 1, dtype=torch.int32)
    if lens:
        cu[1:] = torch.cumsum(torch.tensor(lens, dtype=torch.int64), 0).to(torch.int32)
    CH, HV, dv, dk = wl.CH, wl.HV, wl.dv, wl.dk
    d = {
        "seqlens": lens,
        "cu_seqlens": cu,
        "x": _normal(gen, (T, CH)).to(act),
        "conv_w": _normal(gen, (CH, 4), 0.25).to(act),
        "A_log": torch.rand(HV, generator=gen, dtype=torch.float32) * 2.0 - 1.0,
        "dt_bias": torch.zeros(HV, dtype=torch.float32),
        "u": _normal(gen, (T, HV)).to(act),
        "b_logit": _normal(gen, (T, HV)).to(act),
        "z": _normal(gen, (T, HV * dv)).to(act),
        "norm_w": torch.ones(dv, dtype=torch.float32),
        "state": _normal(gen, (N, HV, dk, dv), 0.02) if wl.init_state else None,
        "conv_state": _normal(gen, (N, CH, 3)).to(act) if wl.init_conv else None,
    }
    S = wl.decode_steps
    if S:
        d["dec_x"] = _normal(gen, (S, N, CH)).to(act)
        d["dec_u"] = _normal(gen, (S, N, HV)).to(act)
        d["dec_b_logit"] = _normal(gen, (S, N, HV)).to(act)
        d["dec_z"] = _normal(gen, (S, N, HV * dv)).to(act)
    return d
