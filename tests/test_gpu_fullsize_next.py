"""The verification round, the Q8 state and the snapshot at the shapes the benchmark runs them:
64 sequences, HK=16, HV=32, dk=dv=128, bf16 inputs, in the benchmark's launch configuration
(one call over the whole batch), checked against the oracle.

- Verification, 8 tokens per sequence: every sequence, on 4 of the 16 q/k heads (first, last and
  two in between) with their v-heads.  Heads never interact, so a head's outputs, checkpoint
  states and histories are the same whether or not the other heads are computed.
- Q8: the encode of the whole 64 x 32-head pool bit for bit, then three Q8 decode steps of the
  whole batch, each against oracle.mixer_decode_q8 from the pool the GPU left after the step
  before, over all heads (the dither is keyed by each code's index in the whole pool, so the
  oracle runs the pool as it is).
- Snapshot: 64 live slots copied to 64 other rows of the same pool, bit for bit."""
import numpy as np
import pytest
import torch

import oracle
from gateddeltanet_linear_attention_gb300 import gdn

from gpu_util import TOL_BF16, rel_max, report

pytestmark = pytest.mark.gpu

N, HK, HV, D = 64, 16, 32, 128
CH = 2 * HK * D + HV * D


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    gdn.load()


def _inputs(rows, seed):
    g = torch.Generator().manual_seed(seed)
    rn = lambda *s, std=1.0: torch.randn(*s, generator=g) * std
    return dict(state=rn(N, HV, D, D, std=0.02), conv=rn(N, CH, 3).to(torch.bfloat16),
                cw=rn(CH, 4, std=0.25).to(torch.bfloat16), A=torch.rand(HV, generator=g) * 2 - 1,
                dt=torch.zeros(HV), nw=torch.ones(D),
                x=rn(rows, CH).to(torch.bfloat16), z=rn(rows, HV * D).to(torch.bfloat16),
                u=rn(rows, HV).to(torch.bfloat16), b=rn(rows, HV).to(torch.bfloat16))


def test_verify_64x8_sampled_heads():
    k = 8
    inp = _inputs(N * k, seed=91)
    slots = N + N * k
    cfg = gdn.make_config(HK, HV, D, D, 64, "bf16", slots)
    st = torch.zeros((slots, HV, D, D), device="cuda"); st[:N] = inp["state"].cuda()
    cv = torch.zeros((slots, CH, 3), dtype=torch.bfloat16, device="cuda"); cv[:N] = inp["conv"].cuda()
    src = torch.arange(N, dtype=torch.int32, device="cuda")
    ckpt = N + k * src
    y = torch.empty((N * k, HV * D), device="cuda")
    ws = torch.empty(gdn.gdn_workspace_size(cfg, N * k, N), dtype=torch.uint8, device="cuda")
    dv = lambda t: t.cuda().contiguous()
    gdn.gdn_mixer_verify(cfg, dv(inp["x"]), dv(inp["z"]), dv(inp["u"]), dv(inp["b"]), dv(inp["cw"]),
                         dv(inp["A"]), dv(inp["dt"]), dv(inp["nw"]), y, st, cv, ckpt, k, ws, state_idx=src)
    torch.cuda.synchronize()
    assert gdn.gdn_device_error() == 0
    kh = [0, 5, 10, HK - 1]
    chs, vh, cols = oracle.head_channels(HK, HV, D, D, kh)
    ry, rs, rc = oracle.mixer_verify(inp["x"][:, chs], inp["cw"][chs], inp["u"][:, vh], inp["b"][:, vh],
                                     inp["A"][vh], inp["dt"][vh], inp["z"][:, cols], inp["nw"], k,
                                     len(kh), len(vh), D, D, inp["state"][:, vh], inp["conv"][:, chs])
    ey = rel_max(y[:, torch.as_tensor(cols, device="cuda")], ry)
    cols_state = st[N:].view(N, k, HV, D, D)[:, :, torch.as_tensor(vh, device="cuda")]
    es = rel_max(cols_state, rs)
    report("verify 64x8 (4 q/k heads)", y=ey, columns=es)
    assert ey <= TOL_BF16 and es <= TOL_BF16, (ey, es)
    got_c = cv[N:].view(N, k, CH, 3)[:, :, torch.as_tensor(chs, device="cuda")].float().cpu().numpy()
    assert np.array_equal(got_c, rc)                                    # raw inputs: exact
    assert torch.equal(st[:N].cpu(), inp["state"])                      # the sources are read only
    assert torch.equal(cv[:N].cpu(), inp["conv"])


def test_q8_pool_encode_and_three_steps():
    steps = 3
    inp = _inputs(N * steps, seed=92)
    cfg = gdn.make_config(HK, HV, D, D, 64, "bf16", N)
    codes = torch.empty((N, HV, D, D), dtype=torch.int8, device="cuda")
    scales = torch.empty((N, HV, D), device="cuda")
    gdn.gdn_state_to_q8(cfg, inp["state"].cuda(), codes, scales, 500)
    torch.cuda.synchronize()
    oc, os_ = oracle.q8_encode(inp["state"].numpy(), 500)
    assert np.array_equal(codes.cpu().numpy(), oc)
    assert np.array_equal(scales.cpu().numpy().view(np.int32), os_.view(np.int32))
    conv = inp["conv"].cuda()
    ws = torch.empty(gdn.gdn_workspace_size(cfg, N, N), dtype=torch.uint8, device="cuda")
    # each step from the pool the GPU left (so that a rare code one step apart does not carry
    # into the next step's comparison): y, the new codes and the history against the oracle
    worst_y, worst_steps, differ = 0.0, 0.0, 0.0
    for t in range(steps):
        rows = slice(t * N, (t + 1) * N)
        gc, gs, gcv = codes.cpu().numpy(), scales.cpu().numpy(), conv.float().cpu().numpy()
        y = torch.empty((N, HV * D), device="cuda")
        gdn.gdn_mixer_decode_q8(cfg, inp["x"][rows].cuda(), inp["z"][rows].cuda(), inp["u"][rows].cuda(),
                                inp["b"][rows].cuda(), inp["cw"].cuda(), inp["A"].cuda(), inp["dt"].cuda(),
                                inp["nw"].cuda(), y, codes, scales, conv, 501 + t, ws)
        torch.cuda.synchronize()
        oy, oc, os_, ocv = oracle.mixer_decode_q8(inp["x"][rows], inp["cw"], inp["u"][rows], inp["b"][rows],
                                                  inp["A"], inp["dt"], inp["z"][rows], inp["nw"], HK, HV, D, D,
                                                  gc, gs, gcv, frame=501 + t)
        worst_y = max(worst_y, rel_max(y, oy))
        deq_g = oracle.q8_decode(codes.cpu().numpy(), scales.cpu().numpy())
        deq_o = oracle.q8_decode(oc, os_)
        step = np.maximum(os_, scales.cpu().numpy())[..., None]
        worst_steps = max(worst_steps, float(np.max(np.abs(deq_g - deq_o) / np.where(step > 0, step, 1))))
        differ = max(differ, float(np.mean(codes.cpu().numpy() != oc)))
        assert np.array_equal(conv.float().cpu().numpy(), ocv)
    assert gdn.gdn_device_error() == 0
    report("q8 64x32 heads, 3 steps", y=worst_y, state_steps=worst_steps, codes_differ=differ)
    assert worst_y <= TOL_BF16 and worst_steps <= 4.0 and differ <= 1e-2


def test_snapshot_64_slots_bitwise():
    g = torch.Generator().manual_seed(93)
    slots = 2 * N
    cfg = gdn.make_config(HK, HV, D, D, 64, "bf16", slots)
    st0 = torch.randn((slots, HV, D, D), generator=g)
    cv0 = torch.randn((slots, CH, 3), generator=g).to(torch.bfloat16)
    st, cv = st0.cuda(), cv0.cuda()
    perm = torch.randperm(N, generator=g)
    src = perm.to(torch.int32)
    dst = torch.arange(N, 2 * N, dtype=torch.int32)
    gdn.gdn_state_copy(cfg, st, cv, st, cv, src.cuda(), dst.cuda())
    torch.cuda.synchronize()
    assert gdn.gdn_device_error() == 0
    es, ec, err = oracle.state_copy(st0.numpy(), cv0.view(torch.int16).numpy(), st0.numpy(),
                                    cv0.view(torch.int16).numpy(), src.numpy(), dst.numpy())
    assert not err
    assert np.array_equal(st.cpu().numpy().view(np.int32), es.view(np.int32))
    assert np.array_equal(cv.cpu().view(torch.int16).numpy(), ec)
