"""Q8 recurrent state on the GPU against the oracle (a quantised state with
error feedback, the DeltaNet Q8 state of the hyperflare release notes: int8
codes with per-row scales, stochastic rounding keyed by a frame counter).

The encoder and decoder are bit-exact against oracle.q8_encode / q8_decode
(every step an fp32 operation rounded to nearest, the same counter-based
dither on both sides).  The Q8 decode step is compared with
oracle.mixer_decode_q8: y within the bf16 tolerance and the decoded state
within a few rounding steps (the two sides round states that differ in the
last fp32 bits, so a code may land one step apart).  A 64-step run against the
fp32 decode reports the drift the quantised state adds."""
import numpy as np
import pytest
import torch

import oracle
from gateddeltanet_linear_attention_gb300 import gdn

from gpu_util import TOL_BF16, rel_max, report

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    gdn.load()


def _inputs(n, HK, HV, d, steps, seed):
    g = torch.Generator().manual_seed(seed)
    rn = lambda *s, std=1.0: (torch.randn(*s, generator=g) * std)
    CH = 2 * HK * d + HV * d
    return dict(
        CH=CH, state=rn(n, HV, d, d, std=0.02), conv=rn(n, CH, 3).to(torch.bfloat16),
        cw=rn(CH, 4, std=0.25).to(torch.bfloat16), A=torch.rand(HV, generator=g) * 2 - 1,
        dt=torch.zeros(HV), nw=torch.ones(d),
        x=[rn(n, CH).to(torch.bfloat16) for _ in range(steps)],
        z=[rn(n, HV * d).to(torch.bfloat16) for _ in range(steps)],
        u=[rn(n, HV).to(torch.bfloat16) for _ in range(steps)],
        b=[rn(n, HV).to(torch.bfloat16) for _ in range(steps)])


@pytest.mark.parametrize("d,frame", [(128, 0), (64, 7), (32, 123456789)])
def test_q8_encode_decode_bitwise(d, frame):
    cfg = gdn.make_config(2, 4, d, d, 64 if d == 128 else 16, "bf16", 3)
    g = torch.Generator().manual_seed(d)
    st = torch.randn((3, 4, d, d), generator=g) * torch.rand((3, 4, d, 1), generator=g) * 2
    st[1, 2, 5] = 0                                                  # a zero row
    codes = torch.empty((3, 4, d, d), dtype=torch.int8, device="cuda")
    scales = torch.empty((3, 4, d), device="cuda")
    gdn.gdn_state_to_q8(cfg, st.cuda(), codes, scales, frame)
    back = torch.empty((3, 4, d, d), device="cuda")
    gdn.gdn_state_from_q8(cfg, codes, scales, back)
    torch.cuda.synchronize()
    ec, es = oracle.q8_encode(st.numpy(), frame)
    assert np.array_equal(codes.cpu().numpy(), ec)
    assert np.array_equal(scales.cpu().numpy().view(np.int32), es.view(np.int32))
    assert np.array_equal(back.cpu().numpy().view(np.int32), oracle.q8_decode(ec, es).view(np.int32))


def _gpu_q8_run(inp, n, HK, HV, d, steps, frame0, state_idx=None, n_slots=None):
    cfg = gdn.make_config(HK, HV, d, d, 64 if d == 128 else 16, "bf16", n_slots or n)
    slots = n_slots or n
    st = torch.zeros((slots, HV, d, d)); st[:n] = inp["state"]
    cv = torch.zeros((slots, inp["CH"], 3), dtype=torch.bfloat16); cv[:n] = inp["conv"]
    codes = torch.empty((slots, HV, d, d), dtype=torch.int8, device="cuda")
    scales = torch.empty((slots, HV, d), device="cuda")
    gdn.gdn_state_to_q8(cfg, st.cuda(), codes, scales, frame0)
    conv = cv.cuda()
    ws = torch.empty(gdn.gdn_workspace_size(cfg, n, n), dtype=torch.uint8, device="cuda")
    si = None if state_idx is None else torch.tensor(state_idx, dtype=torch.int32, device="cuda")
    ys = []
    for t in range(steps):
        y = torch.empty((n, HV * d), device="cuda")
        gdn.gdn_mixer_decode_q8(cfg, inp["x"][t].cuda(), inp["z"][t].cuda(), inp["u"][t].cuda(),
                                inp["b"][t].cuda(), inp["cw"].cuda(), inp["A"].cuda(), inp["dt"].cuda(),
                                inp["nw"].cuda(), y, codes, scales, conv, frame0 + 1 + t, ws, state_idx=si)
        ys.append(y)
    torch.cuda.synchronize()
    return torch.stack(ys), codes, scales, conv


def test_q8_decode_matches_oracle():
    n, HK, HV, d, steps = 3, 2, 4, 128, 6
    inp = _inputs(n, HK, HV, d, steps, seed=41)
    y, codes, scales, conv = _gpu_q8_run(inp, n, HK, HV, d, steps, frame0=10)
    assert gdn.gdn_device_error() == 0
    oc, os_ = oracle.q8_encode(inp["state"].numpy(), 10)
    ocv = oracle._f64(inp["conv"])
    worst_y, worst_steps = 0.0, 0.0
    for t in range(steps):
        oy, oc, os_, ocv = oracle.mixer_decode_q8(inp["x"][t], inp["cw"], inp["u"][t], inp["b"][t], inp["A"],
                                                  inp["dt"], inp["z"][t], inp["nw"], HK, HV, d, d, oc, os_,
                                                  ocv, frame=11 + t)
        worst_y = max(worst_y, rel_max(y[t], oy))
    deq_g = oracle.q8_decode(codes.cpu().numpy(), scales.cpu().numpy())
    deq_o = oracle.q8_decode(oc, os_)
    step = np.maximum(os_, scales.cpu().numpy())[..., None]
    worst_steps = float(np.max(np.abs(deq_g - deq_o) / np.where(step > 0, step, 1)))
    diff_codes = float(np.mean(codes.cpu().numpy() != oc))
    report("q8 decode 6 steps", y=worst_y, state_steps=worst_steps, codes_differ=diff_codes)
    assert worst_y <= TOL_BF16
    assert worst_steps <= 4.0 and diff_codes <= 1e-2
    assert np.array_equal(conv.float().cpu().numpy(), ocv)             # the history: raw inputs


def test_q8_decode_padding_lane_untouched():
    n, HK, HV, d = 3, 2, 4, 64
    inp = _inputs(n, HK, HV, d, 1, seed=42)
    cfg = gdn.make_config(HK, HV, d, d, 16, "bf16", 4)
    y, codes, scales, conv = _gpu_q8_run(inp, n, HK, HV, d, 1, frame0=3, state_idx=[2, -1, 0], n_slots=4)
    assert gdn.gdn_device_error() == 0
    assert torch.all(y[0, 1] == 0)
    st = torch.zeros((4, HV, d, d)); st[:n] = inp["state"]
    ec, es = oracle.q8_encode(st.numpy(), 3)
    assert np.array_equal(codes[1].cpu().numpy(), ec[1]) and np.array_equal(codes[3].cpu().numpy(), ec[3])


def _rms_rel(a, b):
    a = a.detach().double().cpu().numpy() if hasattr(a, "detach") else np.asarray(a, np.float64)
    b = b.detach().double().cpu().numpy() if hasattr(b, "detach") else np.asarray(b, np.float64)
    return float(np.sqrt(np.mean((a - b) ** 2) / np.mean(b * b)))


def test_q8_drift_against_fp32_decode():
    """64 steps from the same state: the Q8 path's y against the fp32 path's.  The rounding
    noise is unbiased, so it is damped by the decay instead of accumulating: the RMS error of y
    over the last 16 steps is no larger (up to sampling noise) than over the first 16."""
    n, HK, HV, d, steps = 4, 2, 4, 128, 64
    inp = _inputs(n, HK, HV, d, steps, seed=43)
    yq, codes, scales, _ = _gpu_q8_run(inp, n, HK, HV, d, steps, frame0=100)
    cfg = gdn.make_config(HK, HV, d, d, 64, "bf16", n)
    st = inp["state"].clone().cuda(); cv = inp["conv"].clone().cuda()
    ws = torch.empty(gdn.gdn_workspace_size(cfg, n, n), dtype=torch.uint8, device="cuda")
    yf = []
    for t in range(steps):
        y = torch.empty((n, HV * d), device="cuda")
        gdn.gdn_mixer_decode(cfg, inp["x"][t].cuda(), inp["z"][t].cuda(), inp["u"][t].cuda(), inp["b"][t].cuda(),
                             inp["cw"].cuda(), inp["A"].cuda(), inp["dt"].cuda(), inp["nw"].cuda(), y, st, cv, ws)
        yf.append(y)
    torch.cuda.synchronize()
    yf = torch.stack(yf)
    first, last = _rms_rel(yq[:16], yf[:16]), _rms_rel(yq[-16:], yf[-16:])
    deq = oracle.q8_decode(codes.cpu().numpy(), scales.cpu().numpy())
    es = _rms_rel(torch.tensor(deq), st)
    report("q8 drift vs fp32 (64 steps, RMS)", y_first16=first, y_last16=last, state=es,
           y_max_abs=max(rel_max(yq[t], yf[t].cpu().numpy()) for t in range(steps)))
    assert first <= 0.05 and last <= 0.05 and es <= 0.05
    assert last <= 2.0 * first + 0.005
