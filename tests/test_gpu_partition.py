"""The multi-GPU split, checked on one GPU: the mixer shards by (sequence,
q/k-head group) with no exchange, so running disjoint shards as separate calls
and putting their results together must reproduce the full call bit for bit.
Two head groups (q/k heads {0, 2} and {1, 3}, each with its v-heads, conv
channels, gates, norm gate columns and state heads gathered into its own
call) and two sequence groups ({0, 2} and {1}, through state_idx into the
shared pool) are compared with one call over everything, for the prefill on
both the tensor-core and the fp32 path and for one decode step."""
import numpy as np
import pytest
import torch

import oracle
from gateddeltanet_linear_attention_gb300 import gdn
from gateddeltanet_linear_attention_gb300.inputs import Workload, make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    gdn.load()


WLS = [
    Workload("part_tc", HK=4, HV=8, dk=128, dv=128, chunk=64, act="bf16", seed=61,
             seqlens=(150, 64, 200), init_state=True, init_conv=True, decode_steps=1),
    Workload("part_simt", HK=4, HV=8, dk=64, dv=64, chunk=16, act="fp32", seed=62,
             seqlens=(40, 17, 70), init_state=True, init_conv=True, decode_steps=1),
]


def _prefill(wl, d, x, z, u, b, cw, A, dt, cu, state, conv, state_idx=None, HK=None, HV=None):
    HK = HK or wl.HK
    HV = HV or wl.HV
    cfg = gdn.make_config(HK, HV, wl.dk, wl.dv, wl.chunk, wl.act, n_slots=state.shape[0])
    T = x.shape[0]
    y = torch.empty((T, HV * wl.dv), device="cuda")
    ws = torch.empty(max(gdn.gdn_workspace_size(cfg, T, cu.shape[0] - 1), 16), dtype=torch.uint8,
                     device="cuda")
    gdn.gdn_mixer_prefill(cfg, x, z, u, b, cw, A, dt, d["norm_w"], cu, y, state_in=state,
                          state_out=state, conv_state=conv, state_idx=state_idx, workspace=ws)
    return y


def _decode(wl, d, x, z, u, b, cw, A, dt, state, conv, HK=None, HV=None):
    HK = HK or wl.HK
    HV = HV or wl.HV
    cfg = gdn.make_config(HK, HV, wl.dk, wl.dv, wl.chunk, wl.act, n_slots=state.shape[0])
    n = x.shape[0]
    y = torch.empty((n, HV * wl.dv), device="cuda")
    ws = torch.empty(gdn.gdn_workspace_size(cfg, n, n), dtype=torch.uint8, device="cuda")
    gdn.gdn_mixer_decode(cfg, x, z, u, b, cw, A, dt, d["norm_w"], y, state, conv, ws)
    return y


@pytest.mark.parametrize("wl", WLS, ids=lambda w: w.name)
def test_head_groups_reproduce_the_full_call(wl):
    d = {k: v.cuda() for k, v in make_inputs(wl).items() if hasattr(v, "cuda")}
    full_state, full_conv = d["state"].clone(), d["conv_state"].clone()
    y_full = _prefill(wl, d, d["x"], d["z"], d["u"], d["b_logit"], d["conv_w"], d["A_log"], d["dt_bias"],
                      d["cu_seqlens"], full_state, full_conv)
    yd_full = _decode(wl, d, d["dec_x"][0], d["dec_z"][0], d["dec_u"][0], d["dec_b_logit"][0], d["conv_w"],
                      d["A_log"], d["dt_bias"], full_state, full_conv)
    torch.cuda.synchronize()
    for group in ([0, 2], [1, 3]):
        chs, vh, cols = (torch.as_tensor(a, device="cuda")
                         for a in oracle.head_channels(wl.HK, wl.HV, wl.dk, wl.dv, group))
        st, cv = d["state"][:, vh].contiguous(), d["conv_state"][:, chs].contiguous()
        kw = dict(HK=len(group), HV=len(vh))
        y = _prefill(wl, d, d["x"][:, chs].contiguous(), d["z"][:, cols].contiguous(),
                     d["u"][:, vh].contiguous(), d["b_logit"][:, vh].contiguous(), d["conv_w"][chs].contiguous(),
                     d["A_log"][vh].contiguous(), d["dt_bias"][vh].contiguous(), d["cu_seqlens"], st, cv, **kw)
        yd = _decode(wl, d, d["dec_x"][0][:, chs].contiguous(), d["dec_z"][0][:, cols].contiguous(),
                     d["dec_u"][0][:, vh].contiguous(), d["dec_b_logit"][0][:, vh].contiguous(),
                     d["conv_w"][chs].contiguous(), d["A_log"][vh].contiguous(), d["dt_bias"][vh].contiguous(),
                     st, cv, **kw)
        torch.cuda.synchronize()
        assert torch.equal(y, y_full[:, cols]), group
        assert torch.equal(yd, yd_full[:, cols]), group
        assert torch.equal(st, full_state[:, vh]) and torch.equal(cv, full_conv[:, chs]), group
    assert gdn.gdn_device_error() == 0


@pytest.mark.parametrize("wl", WLS, ids=lambda w: w.name)
def test_sequence_groups_reproduce_the_full_call(wl):
    d = {k: v.cuda() for k, v in make_inputs(wl).items() if hasattr(v, "cuda")}
    full_state, full_conv = d["state"].clone(), d["conv_state"].clone()
    y_full = _prefill(wl, d, d["x"], d["z"], d["u"], d["b_logit"], d["conv_w"], d["A_log"], d["dt_bias"],
                      d["cu_seqlens"], full_state, full_conv)
    st, cv = d["state"].clone(), d["conv_state"].clone()          # one pool, shared by the shards
    cu = d["cu_seqlens"].cpu().tolist()
    for group in ([0, 2], [1]):
        rows = torch.cat([torch.arange(cu[n], cu[n + 1]) for n in group]).cuda()
        lens = [cu[n + 1] - cu[n] for n in group]
        cu_g = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32, device="cuda")
        y = _prefill(wl, d, d["x"][rows].contiguous(), d["z"][rows].contiguous(), d["u"][rows].contiguous(),
                     d["b_logit"][rows].contiguous(), d["conv_w"], d["A_log"], d["dt_bias"], cu_g, st, cv,
                     state_idx=torch.tensor(group, dtype=torch.int32, device="cuda"))
        torch.cuda.synchronize()
        assert torch.equal(y, y_full[rows]), group
    assert torch.equal(st, full_state) and torch.equal(cv, full_conv)
    assert gdn.gdn_device_error() == 0
