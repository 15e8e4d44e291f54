"""Q8 recurrent state on the GPU against the oracle (the DeltaNet Q8 state of
the warpfront/hipfire PR #527 thread: int8 codes with per-row scales,
stochastic requantisation with a dither keyed by a frame counter, and an
optional error-feedback residual).

The encoder and decoder are bit-exact against oracle.q8_encode / q8_decode
(every step an fp32 operation rounded to nearest, the same counter-based
dither on both sides), with and without the residual.  The Q8 decode step is
compared with oracle.mixer_decode_q8: y within the bf16 tolerance and the
decoded state (plus residual) within a few rounding steps (the two sides
round states that differ in the last fp32 bits, so a code may land one step
apart).  A 256-step run against the fp32 decode reports the drift the
quantised state adds, with and without error feedback."""
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


@pytest.mark.parametrize("ef", [False, True])
@pytest.mark.parametrize("d,frame", [(128, 0), (64, 7), (32, 123456789)])
def test_q8_encode_decode_bitwise(d, frame, ef):
    cfg = gdn.make_config(2, 4, d, d, 64 if d == 128 else 16, "bf16", 3)
    g = torch.Generator().manual_seed(d)
    st = torch.randn((3, 4, d, d), generator=g) * torch.rand((3, 4, d, 1), generator=g) * 2
    st[1, 2, 5] = 0                                                  # a zero row
    codes = torch.empty((3, 4, d, d), dtype=torch.int8, device="cuda")
    scales = torch.empty((3, 4, d), device="cuda")
    res = torch.full((3, 4, d, d), float("nan"), dtype=torch.bfloat16, device="cuda") if ef else None
    gdn.gdn_state_to_q8(cfg, st.cuda(), codes, scales, frame, residual=res)
    back = torch.empty((3, 4, d, d), device="cuda")
    gdn.gdn_state_from_q8(cfg, codes, scales, back)
    torch.cuda.synchronize()
    if ef:
        ec, es, er = oracle.q8_encode(st.numpy(), frame, residual=np.zeros(st.shape, np.float32))
        assert np.array_equal(res.float().cpu().numpy().view(np.int32), er.view(np.int32))
    else:
        ec, es = oracle.q8_encode(st.numpy(), frame)
    assert np.array_equal(codes.cpu().numpy(), ec)
    assert np.array_equal(scales.cpu().numpy().view(np.int32), es.view(np.int32))
    assert np.array_equal(back.cpu().numpy().view(np.int32), oracle.q8_decode(ec, es).view(np.int32))


def _gpu_q8_run(inp, n, HK, HV, d, steps, frame0, state_idx=None, n_slots=None, ef=False):
    cfg = gdn.make_config(HK, HV, d, d, 64 if d == 128 else 16, "bf16", n_slots or n)
    slots = n_slots or n
    st = torch.zeros((slots, HV, d, d)); st[:n] = inp["state"]
    cv = torch.zeros((slots, inp["CH"], 3), dtype=torch.bfloat16); cv[:n] = inp["conv"]
    codes = torch.empty((slots, HV, d, d), dtype=torch.int8, device="cuda")
    scales = torch.empty((slots, HV, d), device="cuda")
    res = torch.empty((slots, HV, d, d), dtype=torch.bfloat16, device="cuda") if ef else None
    gdn.gdn_state_to_q8(cfg, st.cuda(), codes, scales, frame0, residual=res)
    conv = cv.cuda()
    ws = torch.empty(gdn.gdn_workspace_size(cfg, n, n), dtype=torch.uint8, device="cuda")
    si = None if state_idx is None else torch.tensor(state_idx, dtype=torch.int32, device="cuda")
    ys = []
    for t in range(steps):
        y = torch.empty((n, HV * d), device="cuda")
        gdn.gdn_mixer_decode_q8(cfg, inp["x"][t].cuda(), inp["z"][t].cuda(), inp["u"][t].cuda(),
                                inp["b"][t].cuda(), inp["cw"].cuda(), inp["A"].cuda(), inp["dt"].cuda(),
                                inp["nw"].cuda(), y, codes, scales, conv, frame0 + 1 + t, ws, state_idx=si,
                                residual=res)
        ys.append(y)
    torch.cuda.synchronize()
    out = (torch.stack(ys), codes, scales, conv)
    return out + (res,) if ef else out


@pytest.mark.parametrize("ef", [False, True])
def test_q8_decode_matches_oracle(ef):
    n, HK, HV, d, steps = 3, 2, 4, 128, 6
    inp = _inputs(n, HK, HV, d, steps, seed=41)
    got = _gpu_q8_run(inp, n, HK, HV, d, steps, frame0=10, ef=ef)
    y, codes, scales, conv = got[:4]
    assert gdn.gdn_device_error() == 0
    if ef:
        oc, os_, ores = oracle.q8_encode(inp["state"].numpy(), 10, residual=np.zeros((n, HV, d, d), np.float32))
    else:
        oc, os_ = oracle.q8_encode(inp["state"].numpy(), 10)
        ores = None
    ocv = oracle._f64(inp["conv"])
    worst_y = 0.0
    for t in range(steps):
        out = oracle.mixer_decode_q8(inp["x"][t], inp["cw"], inp["u"][t], inp["b"][t], inp["A"], inp["dt"],
                                     inp["z"][t], inp["nw"], HK, HV, d, d, oc, os_, ocv, frame=11 + t,
                                     residual=ores)
        oy, oc, os_, ocv = out[:4]
        if ef:
            ores = out[4]
        worst_y = max(worst_y, rel_max(y[t], oy))
    deq_g = oracle.q8_decode(codes.cpu().numpy(), scales.cpu().numpy())
    deq_o = oracle.q8_decode(oc, os_)
    step = np.maximum(os_, scales.cpu().numpy())[..., None]
    steps_off = np.abs(deq_g - deq_o) / np.where(step > 0, step, 1)
    worst_steps = float(np.max(steps_off))
    diff_codes = float(np.mean(codes.cpu().numpy() != oc))
    extra = {}
    if ef:
        # what the pool represents, codes plus residual, agrees far below one step
        res_g = got[4].float().cpu().numpy()
        carried = np.abs((deq_g + res_g) - (deq_o + ores)) / np.where(step > 0, step, 1)
        extra = dict(carried_steps_max=float(np.max(carried)), carried_steps_mean=float(np.mean(carried)))
        assert float(np.mean(carried)) <= 1e-2
    report("q8%s decode 6 steps" % (" EF" if ef else ""), y=worst_y, state_steps=worst_steps,
           codes_differ=diff_codes, **extra)
    assert worst_y <= TOL_BF16
    assert worst_steps <= 4.0 and diff_codes <= 1e-2
    assert np.array_equal(conv.float().cpu().numpy(), ocv)             # the history: raw inputs


@pytest.mark.parametrize("d", [64, 128])   # (at 128 the encode runs on its own warps)
def test_q8_decode_padding_lane_untouched(d):
    n, HK, HV = 3, 2, 4
    inp = _inputs(n, HK, HV, d, 1, seed=42)
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
    """256 steps from the same state: the Q8 path's y and state against the fp32 path's, with and
    without error feedback.  The rounding noise is unbiased, so it is damped by the decay instead
    of accumulating: in both forms the RMS error of y over the last 64 steps is no larger (up to
    sampling noise) than over the first 64, and the state stays within a few percent.  Whether
    feedback lowers the error depends on the decay (it moves the noise to high frequencies, which
    a strong decay passes about as easily as white noise); both figures are reported."""
    n, HK, HV, d, steps = 4, 2, 4, 128, 256
    inp = _inputs(n, HK, HV, d, steps, seed=43)
    yq, codes, scales, _ = _gpu_q8_run(inp, n, HK, HV, d, steps, frame0=100)
    ye, codes_e, scales_e, _, res_e = _gpu_q8_run(inp, n, HK, HV, d, steps, frame0=100, ef=True)
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
    assert gdn.gdn_device_error() == 0
    yf = torch.stack(yf)
    out = {}
    for tag, yy, cc, ss in (("plain", yq, codes, scales), ("ef", ye, codes_e, scales_e)):
        deq = oracle.q8_decode(cc.cpu().numpy(), ss.cpu().numpy())
        out[tag] = dict(first64=_rms_rel(yy[:64], yf[:64]), last64=_rms_rel(yy[-64:], yf[-64:]),
                        state=_rms_rel(torch.tensor(deq), st),
                        y_max=max(rel_max(yy[t], yf[t].cpu().numpy()) for t in range(steps)))
    report("q8 drift vs fp32 decode (256 steps, RMS-relative)",
           **{f"{k}_{m}": v for k, d_ in out.items() for m, v in d_.items()})
    for r in out.values():
        assert r["first64"] <= 0.05 and r["last64"] <= 0.05 and r["state"] <= 0.05
        assert r["last64"] <= 2.0 * r["first64"] + 0.005
