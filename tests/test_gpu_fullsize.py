"""The four full-size bf16 workloads, run on the GPU exactly as the benchmark
launches them (the fused prefill / decode entry points over the whole batch),
checked against the oracle: prefill_8k on every head; varlen_16, long_64k and
decode_64x256 on 8 of the 16 q/k heads (first, last, odd and middle ones) and
all their v-heads.  Heads never interact, so a sampled head's outputs and
state are the same whether or not the other heads are computed."""
import numpy as np
import pytest
import torch

from gateddeltanet_linear_attention_gb300 import gdn
from gateddeltanet_linear_attention_gb300.inputs import WORKLOADS, make_inputs

from gpu_util import TOL_BF16, GpuMixer, head_channels, oracle_mixer, rel_max, report, vcols

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    gdn.load()


def _cmp(wl, y_gpu, ref, kheads, state_gpu=None, what=""):
    _, vh = head_channels(wl, kheads)
    cols = vcols(wl, vh)
    ey = rel_max(y_gpu[:, torch.as_tensor(cols, device=y_gpu.device)], ref["y"])
    es = None
    if state_gpu is not None:
        es = rel_max(state_gpu[:, torch.as_tensor(vh, device=state_gpu.device)], ref["state"])
    report(what, y=ey, state=es if es is not None else float("nan"))
    assert ey <= TOL_BF16, (what, "y", ey)
    if es is not None:
        assert es <= TOL_BF16, (what, "state", es)
    return ey


def test_prefill_8k():
    wl = WORKLOADS["prefill_8k"]
    inp = make_inputs(wl)
    m = GpuMixer(wl, inp)
    y = m.prefill()
    torch.cuda.synchronize()
    assert gdn.gdn_device_error() == 0
    kh = list(range(wl.HK))
    ref = oracle_mixer(wl, inp, kheads=kh)
    _cmp(wl, y, ref, kh, m.state, "prefill_8k (all heads)")


def test_varlen_16():
    wl = WORKLOADS["varlen_16"]
    inp = make_inputs(wl)
    m = GpuMixer(wl, inp)
    y = m.prefill()
    torch.cuda.synchronize()
    assert gdn.gdn_device_error() == 0
    kh = [0, 1, 3, 6, 7, 9, 12, wl.HK - 1]
    ref = oracle_mixer(wl, inp, kheads=kh)
    _cmp(wl, y, ref, kh, m.state, "varlen_16 (8 q/k heads)")
    chs, _ = head_channels(wl, kh)
    assert torch.equal(m.conv[:, torch.as_tensor(chs, device="cuda")].float().cpu(),
                       torch.tensor(ref["conv_state"], dtype=torch.float32))


def test_decode_64x256():
    wl = WORKLOADS["decode_64x256"]
    inp = make_inputs(wl)
    m = GpuMixer(wl, inp)
    N = wl.n_decode
    cu = np.arange(N + 1, dtype=np.int32)
    kh = [0, 3, 5, 6, 9, 10, 12, wl.HK - 1]
    chs, vh = head_channels(wl, kh)
    st, cs = inp["state"][:, torch.as_tensor(vh)], inp["conv_state"][:, torch.as_tensor(chs)]
    worst = 0.0
    ys = []
    for t in range(wl.decode_steps):
        ys.append(m.decode(inp["dec_x"][t].cuda(), inp["dec_z"][t].cuda(), inp["dec_u"][t].cuda(),
                           inp["dec_b_logit"][t].cuda()))
    torch.cuda.synchronize()
    assert gdn.gdn_device_error() == 0
    # oracle on the sampled heads (state and history already sliced to them)
    sub = dict(inp)
    sub["conv_w"] = inp["conv_w"][torch.as_tensor(chs)]
    sub["A_log"], sub["dt_bias"] = inp["A_log"][torch.as_tensor(vh)], inp["dt_bias"][torch.as_tensor(vh)]
    from gateddeltanet_linear_attention_gb300.inputs import shrink
    wl_s = shrink(wl, HK=len(kh), HV=len(vh))
    cols = vcols(wl, vh)
    for t in range(wl.decode_steps):
        ref = oracle_mixer(wl_s, sub, x=inp["dec_x"][t][:, torch.as_tensor(chs)],
                           u=inp["dec_u"][t][:, torch.as_tensor(vh)],
                           b=inp["dec_b_logit"][t][:, torch.as_tensor(vh)],
                           z=inp["dec_z"][t][:, torch.as_tensor(cols)], cu=cu, state=st,
                           conv_state=cs)
        st, cs = torch.tensor(ref["state"]), torch.tensor(ref["conv_state"])
        worst = max(worst, rel_max(ys[t][:, torch.as_tensor(cols, device="cuda")], ref["y"]))
    es = rel_max(m.state[:, torch.as_tensor(vh, device="cuda")], ref["state"])
    report("decode_64x256", y_worst_step=worst, state=es)
    assert worst <= TOL_BF16, ("decode y", worst)
    assert es <= TOL_BF16, ("decode state", es)


def test_long_64k_then_512_decode_steps():
    wl = WORKLOADS["long_64k"]
    inp = make_inputs(wl)
    m = GpuMixer(wl, inp)
    y = m.prefill()
    state_after_prefill = m.state.clone()
    ys = []
    for t in range(wl.decode_steps):
        ys.append(m.decode(inp["dec_x"][t].cuda(), inp["dec_z"][t].cuda(), inp["dec_u"][t].cuda(),
                           inp["dec_b_logit"][t].cuda()))
    torch.cuda.synchronize()
    assert gdn.gdn_device_error() == 0
    kh = [0, 2, 5, 7, 8, 11, 13, wl.HK - 1]
    ref = oracle_mixer(wl, inp, kheads=kh)
    _cmp(wl, y, ref, kh, state_after_prefill, "long_64k prefill (8 q/k heads)")
    chs, vh = head_channels(wl, kh)
    cols = vcols(wl, vh)
    from gateddeltanet_linear_attention_gb300.inputs import shrink
    wl_s = shrink(wl, HK=len(kh), HV=len(vh))
    sub = dict(inp)
    sub["conv_w"] = inp["conv_w"][torch.as_tensor(chs)]
    sub["A_log"], sub["dt_bias"] = inp["A_log"][torch.as_tensor(vh)], inp["dt_bias"][torch.as_tensor(vh)]
    st, cs = torch.tensor(ref["state"]), torch.tensor(ref["conv_state"])
    cu = np.array([0, 1], np.int32)
    yd = []
    for t in range(wl.decode_steps):
        r = oracle_mixer(wl_s, sub, x=inp["dec_x"][t][:, torch.as_tensor(chs)],
                         u=inp["dec_u"][t][:, torch.as_tensor(vh)],
                         b=inp["dec_b_logit"][t][:, torch.as_tensor(vh)],
                         z=inp["dec_z"][t][:, torch.as_tensor(cols)], cu=cu, state=st,
                         conv_state=cs)
        st, cs = torch.tensor(r["state"]), torch.tensor(r["conv_state"])
        yd.append(r["y"])
    ey = rel_max(torch.cat(ys)[:, torch.as_tensor(cols, device="cuda")], np.concatenate(yd))
    es = rel_max(m.state[:, torch.as_tensor(vh, device="cuda")], r["state"])
    report("long_64k decode", y=ey, state=es)
    assert ey <= TOL_BF16, ("long decode y", ey)
    assert es <= TOL_BF16, ("long final state", es)
