"""CUDA graph capture of the fused entry points (the interface list's capture
safety: no allocation, no synchronisation and no host read of device data
inside a call).  A prefill followed by three decode steps, a verification
round, a snapshot and a Q8 decode step are captured into one graph after an
eager warm-up; replaying the graph from the same initial buffers reproduces
the eager results bit for bit."""
import pytest
import torch

from gateddeltanet_linear_attention_gb300 import gdn
from gateddeltanet_linear_attention_gb300.inputs import Workload, make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    gdn.load()


def test_graph_replay_is_bitwise_eager():
    wl = Workload("g", HK=2, HV=4, dk=128, dv=128, chunk=64, act="bf16", seed=51, seqlens=(100, 37),
                  init_state=True, init_conv=True, decode_steps=3)
    inp = make_inputs(wl)
    N, k = 2, 4
    slots = N + N * k + N                       # live, verification columns, snapshots
    cfg = gdn.make_config(wl.HK, wl.HV, wl.dk, wl.dv, wl.chunk, wl.act, n_slots=slots)
    d = {kk: v.cuda() for kk, v in inp.items() if hasattr(v, "cuda")}
    T = d["x"].shape[0]
    st0 = torch.zeros((slots, wl.HV, wl.dk, wl.dv), device="cuda"); st0[:N] = d["state"]
    cv0 = torch.zeros((slots, wl.CH, 3), dtype=torch.bfloat16, device="cuda"); cv0[:N] = d["conv_state"]
    state, conv = st0.clone(), cv0.clone()
    codes = torch.zeros((slots, wl.HV, wl.dk, wl.dv), dtype=torch.int8, device="cuda")
    scales = torch.zeros((slots, wl.HV, wl.dk), device="cuda")
    ws = torch.empty(gdn.gdn_workspace_size(cfg, max(T, N * k), N), dtype=torch.uint8, device="cuda")
    y = torch.empty((T, wl.HV * wl.dv), device="cuda")
    yd = [torch.empty((N, wl.HV * wl.dv), device="cuda") for _ in range(3)]
    yv = torch.empty((N * k, wl.HV * wl.dv), device="cuda")
    yq = torch.empty((N, wl.HV * wl.dv), device="cuda")
    live = torch.arange(N, dtype=torch.int32, device="cuda")
    ckpt = torch.tensor([N, N + k], dtype=torch.int32, device="cuda")
    snap = torch.arange(N + N * k, slots, dtype=torch.int32, device="cuda")
    xv = d["x"][:N * k].contiguous(); zv = d["z"][:N * k].contiguous()
    uv = d["u"][:N * k].contiguous(); bv = d["b_logit"][:N * k].contiguous()
    common = (d["conv_w"], d["A_log"], d["dt_bias"], d["norm_w"])

    def body():
        gdn.gdn_mixer_prefill(cfg, d["x"], d["z"], d["u"], d["b_logit"], *common, d["cu_seqlens"], y,
                              state_in=state, state_out=state, conv_state=conv, state_idx=live,
                              workspace=ws)
        for t in range(3):
            gdn.gdn_mixer_decode(cfg, d["dec_x"][t], d["dec_z"][t], d["dec_u"][t], d["dec_b_logit"][t],
                                 *common, yd[t], state, conv, ws, state_idx=live)
        gdn.gdn_mixer_verify(cfg, xv, zv, uv, bv, *common, yv, state, conv, ckpt, k, ws, state_idx=live)
        gdn.gdn_state_copy(cfg, state, conv, state, conv, live, snap)
        gdn.gdn_state_to_q8(cfg, state, codes, scales, 7)
        gdn.gdn_mixer_decode_q8(cfg, d["dec_x"][0], d["dec_z"][0], d["dec_u"][0], d["dec_b_logit"][0],
                                *common, yq, codes, scales, conv, 8, ws, state_idx=live)

    body()                                      # eager (also resolves the device error word)
    torch.cuda.synchronize()
    assert gdn.gdn_device_error() == 0
    eager = [t.clone() for t in [y, *yd, yv, yq, state, conv, codes, scales]]

    state.copy_(st0); conv.copy_(cv0); codes.zero_(); scales.zero_()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            body()
    torch.cuda.current_stream().wait_stream(s)
    state.copy_(st0); conv.copy_(cv0); codes.zero_(); scales.zero_()
    for b in (y, *yd, yv, yq):
        b.fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    assert gdn.gdn_device_error() == 0
    for got, ref in zip([y, *yd, yv, yq, state, conv, codes, scales], eager):
        assert torch.equal(got, ref)
