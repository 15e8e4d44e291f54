"""Helpers shared by the GPU tests: run the CUDA path through the C ABI and the
oracle on the same seeded inputs, slice a workload down to a subset of heads
(heads are independent, so the oracle can check a sample of a full-size run),
and the parity metric max|delta| / RMS(oracle)."""
import numpy as np
import torch

import oracle
from gateddeltanet_linear_attention_gb300 import gdn

TOL_BF16 = 1e-2      # max|delta|/RMS(oracle) on outputs, bf16 inputs
TOL_FP32 = 1e-4      # same, fp32-input mode, outputs and final state


def rel_max(gpu, ref):
    """max |gpu - ref| / RMS(ref), over the whole tensor."""
    g = gpu.detach().double().cpu().numpy() if hasattr(gpu, "detach") else np.asarray(gpu, np.float64)
    r = np.asarray(ref, np.float64)
    assert g.shape == r.shape, (g.shape, r.shape)
    rms = np.sqrt(np.mean(r * r))
    if rms == 0:
        return float(np.abs(g).max()) if g.size else 0.0
    return float(np.abs(g - r).max() / rms)


def report(name, **errs):
    """Print measured parity errors (visible with pytest -s)."""
    print("PARITY %-40s %s" % (name, " ".join("%s=%.3e" % kv for kv in errs.items())), flush=True)


def dev(t, device="cuda"):
    return None if t is None else t.to(device).contiguous()


def cfg_for(wl, n_slots):
    return gdn.make_config(wl.HK, wl.HV, wl.dk, wl.dv, wl.chunk, wl.act, n_slots)


def head_channels(wl, kheads):
    """Channel indices (into CH) and v-head indices for a subset of q/k heads."""
    chs, vh, _ = oracle.head_channels(wl.HK, wl.HV, wl.dk, wl.dv, kheads)
    return chs, vh


def vcols(wl, vheads):
    return np.array([h * wl.dv + j for h in vheads for j in range(wl.dv)])


def oracle_mixer(wl, inp, kheads=None, prefix="", x=None, u=None, b=None, z=None, cu=None,
                 state=None, conv_state=None, slot_idx=None, dumps=False, n_threads=None):
    """Run the oracle on (a head subset of) a workload's inputs (full-width tensors, sliced to
    the subset by oracle.mixer_heads)."""
    kheads = list(range(wl.HK)) if kheads is None else list(kheads)
    x = inp[prefix + "x"] if x is None else x
    u = inp[prefix + "u"] if u is None else u
    b = inp[prefix + "b_logit"] if b is None else b
    z = inp[prefix + "z"] if z is None else z
    st = inp["state"] if state is None else state
    cs = inp["conv_state"] if conv_state is None else conv_state
    cu = inp["cu_seqlens"] if cu is None else cu
    return oracle.mixer_heads(x, inp["conv_w"], u, b, inp["A_log"], inp["dt_bias"], z, inp["norm_w"], cu,
                              wl.HK, wl.HV, wl.dk, wl.dv, kheads, state=st, conv_state=cs,
                              slot_idx=slot_idx, dumps=dumps, n_threads=n_threads)


class GpuMixer:
    """The CUDA path of one workload through the C ABI (device-resident)."""

    def __init__(self, wl, inp, n_slots=None, y_dtype=torch.float32, state_idx=None):
        self.wl = wl
        N = len(inp["seqlens"]) if inp["seqlens"] else wl.n_decode
        self.n_slots = n_slots or max(N, 1)
        self.cfg = cfg_for(wl, self.n_slots)
        self.inp = inp
        d = {k: dev(v) for k, v in inp.items() if hasattr(v, "to")}
        self.d = d
        self.y_dtype = y_dtype
        self.state_idx = dev(state_idx)
        if inp["state"] is not None:
            self.state = d["state"].clone()
        else:
            self.state = torch.zeros((self.n_slots, wl.HV, wl.dk, wl.dv), device="cuda")
        if inp["conv_state"] is not None:
            self.conv = d["conv_state"].clone()
        else:
            self.conv = torch.zeros((self.n_slots, wl.CH, 3), dtype=wl.torch_act, device="cuda")

    def prefill(self, x=None, z=None, u=None, b=None, cu=None):
        d = self.d
        x = d["x"] if x is None else x
        z = d["z"] if z is None else z
        u = d["u"] if u is None else u
        b = d["b_logit"] if b is None else b
        cu = d["cu_seqlens"] if cu is None else cu
        T = x.shape[0]
        ws = torch.empty(max(gdn.gdn_workspace_size(self.cfg, T, cu.shape[0] - 1), 16),
                         dtype=torch.uint8, device="cuda")
        y = torch.empty((T, self.wl.HV * self.wl.dv), dtype=self.y_dtype, device="cuda")
        gdn.gdn_mixer_prefill(self.cfg, x, z, u, b, d["conv_w"], d["A_log"], d["dt_bias"],
                              d["norm_w"], cu, y, state_in=self.state, state_out=self.state,
                              conv_state=self.conv, state_idx=self.state_idx, workspace=ws)
        return y

    def decode(self, x, z, u, b):
        d = self.d
        n = x.shape[0]
        y = torch.empty((n, self.wl.HV * self.wl.dv), dtype=self.y_dtype, device="cuda")
        if getattr(self, "_dec_ws", None) is None or self._dec_ws.numel() < gdn.gdn_workspace_size(
                self.cfg, n, n):
            self._dec_ws = torch.empty(gdn.gdn_workspace_size(self.cfg, n, n), dtype=torch.uint8,
                                       device="cuda")
        gdn.gdn_mixer_decode(self.cfg, x, z, u, b, d["conv_w"], d["A_log"], d["dt_bias"],
                             d["norm_w"], y, self.state, self.conv, self._dec_ws,
                             state_idx=self.state_idx)
        return y
