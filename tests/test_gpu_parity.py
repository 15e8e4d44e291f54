"""Parity of the CUDA path (through the C ABI) with the fp64 oracle.

Small and ragged cases are compared element by element over every output;
the full-size workloads run exactly as the benchmark launches them and are
compared on a sample of heads that the oracle recomputes (heads are
independent).  Gate: max|delta| / RMS(oracle) <= 1e-2 for bf16 inputs and
<= 1e-4 (outputs and final state) in fp32-input mode.
"""
import numpy as np
import pytest
import torch

import oracle
from gateddeltanet_linear_attention_gb300 import gdn
from gateddeltanet_linear_attention_gb300.inputs import WORKLOADS, Workload, make_inputs, shrink

from gpu_util import (TOL_BF16, TOL_FP32, GpuMixer, dev, head_channels, oracle_mixer, rel_max,
                      report, vcols)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    gdn.load()


def _check_prefill(wl, inp, tol, y_dtype=torch.float32, state_idx=None, slot_idx=None, n_slots=None):
    m = GpuMixer(wl, inp, y_dtype=y_dtype, state_idx=state_idx, n_slots=n_slots)
    y = m.prefill()
    ref = oracle_mixer(wl, inp, slot_idx=slot_idx,
                       state=None if inp["state"] is None else inp["state"][:m.n_slots],
                       conv_state=None if inp["conv_state"] is None else inp["conv_state"][:m.n_slots])
    torch.cuda.synchronize()
    assert gdn.gdn_device_error() == 0
    ey = rel_max(y, ref["y"])
    es = rel_max(m.state, ref["state"])
    report(wl.name + str(inp["seqlens"])[:30], y=ey, state=es)
    assert ey <= tol, ("y", ey)
    assert es <= tol, ("state", es)
    if wl.act == "bf16":
        # the conv history is a copy of raw inputs: exact
        assert torch.equal(m.conv.float().cpu(), torch.tensor(ref["conv_state"], dtype=torch.float32))
    else:
        assert rel_max(m.conv, ref["conv_state"]) == 0.0
    return m, y, ref


def test_tiny_fp32_workload():
    wl = WORKLOADS["tiny_fp32"]
    _check_prefill(wl, make_inputs(wl), TOL_FP32)


@pytest.mark.parametrize("d,chunk,HK,HV", [(32, 16, 2, 2), (64, 16, 2, 4), (128, 64, 2, 4),
                                           (128, 64, 1, 4), (64, 64, 4, 4), (128, 16, 2, 2)])
def test_fp32_mode_shapes(d, chunk, HK, HV):
    wl = Workload("t", HK=HK, HV=HV, dk=d, dv=d, chunk=chunk, act="fp32", seed=11,
                  seqlens=(1, 77, 0, 130), init_state=True, init_conv=True)
    _check_prefill(wl, make_inputs(wl), TOL_FP32)


@pytest.mark.parametrize("lens", [(300,), (63, 64, 65, 1, 0, 129)])
def test_bf16_prefill_ragged(lens):
    wl = Workload("t", HK=4, HV=8, dk=128, dv=128, chunk=64, act="bf16", seed=12, seqlens=lens,
                  init_state=True, init_conv=True)
    _check_prefill(wl, make_inputs(wl), TOL_BF16)


def test_bf16_tensor_core_many_short_sequences():
    # 300 sequences (more than the 256-way chunk search of the parallel kernel covers in one
    # round), lengths 0 .. 70 including empty and one-token ones
    rng = np.random.default_rng(5)
    lens = tuple(int(x) for x in rng.integers(0, 71, size=300))
    lens = (0, 1) + lens[2:]
    wl = Workload("many", HK=1, HV=2, dk=128, dv=128, chunk=64, act="bf16", seed=16, seqlens=lens,
                  init_state=True, init_conv=True)
    _check_prefill(wl, make_inputs(wl), TOL_BF16)


def test_bf16_tensor_core_padding_lane():
    lens = (5, 0, 70, 3, 130)
    wl = Workload("t", HK=2, HV=4, dk=128, dv=128, chunk=64, act="bf16", seed=17, seqlens=lens,
                  init_state=True, init_conv=True)
    inp = make_inputs(wl)
    smap = torch.tensor([4, 2, -1, 0, 1], dtype=torch.int32)   # lane 2 is padding; slot 3 unused
    m = GpuMixer(wl, inp, state_idx=smap, n_slots=5)
    y = m.prefill()
    torch.cuda.synchronize()
    assert gdn.gdn_device_error() == 0
    ref = oracle_mixer(wl, inp, slot_idx=smap.numpy())
    cu = inp["cu_seqlens"]
    ey, es = rel_max(y, ref["y"]), rel_max(m.state, ref["state"])
    report("tc padding lane", y=ey, state=es)
    assert ey <= TOL_BF16 and es <= TOL_BF16
    assert torch.count_nonzero(y[cu[2]:cu[3]]) == 0
    torch.testing.assert_close(m.state[3].cpu(), inp["state"][3], rtol=0, atol=0)  # untouched


def test_bf16_y_is_rounded_fp32_y():
    wl = Workload("t", HK=2, HV=4, dk=128, dv=128, chunk=64, act="bf16", seed=13, seqlens=(150,),
                  init_state=True, init_conv=True)
    inp = make_inputs(wl)
    y32 = GpuMixer(wl, inp).prefill()
    y16 = GpuMixer(wl, inp, y_dtype=torch.bfloat16).prefill()
    assert torch.equal(y16, y32.to(torch.bfloat16))


def test_slot_map_padding_lane_and_empty_sequences():
    lens = (5, 0, 70, 3, 17)
    wl = Workload("t", HK=2, HV=4, dk=64, dv=64, chunk=16, act="bf16", seed=14, seqlens=lens,
                  init_state=True, init_conv=True)
    inp = make_inputs(wl)
    smap = torch.tensor([4, 2, -1, 0, 1], dtype=torch.int32)   # lane 2 is padding; slot 3 unused
    m = GpuMixer(wl, inp, state_idx=smap, n_slots=5)
    y = m.prefill()
    ref = oracle_mixer(wl, inp, slot_idx=smap.numpy())
    cu = inp["cu_seqlens"]
    assert rel_max(y, ref["y"]) <= TOL_BF16
    assert torch.count_nonzero(y[cu[2]:cu[3]]) == 0
    assert rel_max(m.state, ref["state"]) <= TOL_BF16
    torch.testing.assert_close(m.state[3].cpu(), inp["state"][3], rtol=0, atol=0)  # untouched
    assert torch.equal(m.conv.float().cpu(), torch.tensor(ref["conv_state"], dtype=torch.float32))


def test_decode_steps_small():
    wl = Workload("t", HK=2, HV=4, dk=128, dv=128, chunk=64, act="bf16", seed=15, init_state=True,
                  init_conv=True, decode_steps=6, n_decode=5)
    inp = make_inputs(wl)
    m = GpuMixer(wl, inp)
    st, cs = inp["state"], inp["conv_state"]
    cu = torch.arange(6, dtype=torch.int32)
    for t in range(6):
        y = m.decode(dev(inp["dec_x"][t]), dev(inp["dec_z"][t]), dev(inp["dec_u"][t]),
                     dev(inp["dec_b_logit"][t]))
        ref = oracle_mixer(wl, inp, x=inp["dec_x"][t], u=inp["dec_u"][t], b=inp["dec_b_logit"][t],
                           z=inp["dec_z"][t], cu=cu, state=st, conv_state=cs)
        st, cs = torch.tensor(ref["state"]), torch.tensor(ref["conv_state"])
        assert rel_max(y, ref["y"]) <= TOL_BF16
    assert rel_max(m.state, ref["state"]) <= TOL_BF16
    assert torch.equal(m.conv.float().cpu(), torch.tensor(ref["conv_state"], dtype=torch.float32))


def test_decode_fp32_and_gqa4():
    wl = Workload("t", HK=1, HV=4, dk=64, dv=64, chunk=16, act="fp32", seed=16, init_state=True,
                  init_conv=True, decode_steps=3, n_decode=3)
    inp = make_inputs(wl)
    m = GpuMixer(wl, inp)
    st, cs = inp["state"], inp["conv_state"]
    cu = torch.arange(4, dtype=torch.int32)
    for t in range(3):
        y = m.decode(dev(inp["dec_x"][t]), dev(inp["dec_z"][t]), dev(inp["dec_u"][t]),
                     dev(inp["dec_b_logit"][t]))
        ref = oracle_mixer(wl, inp, x=inp["dec_x"][t], u=inp["dec_u"][t], b=inp["dec_b_logit"][t],
                           z=inp["dec_z"][t], cu=cu, state=st, conv_state=cs)
        st, cs = torch.tensor(ref["state"]), torch.tensor(ref["conv_state"])
        assert rel_max(y, ref["y"]) <= TOL_FP32
    assert rel_max(m.state, ref["state"]) <= TOL_FP32


def test_prefill_then_decode_matches_one_oracle_pass():
    """Continuation: prefill of T1 tokens, then one-token decode steps == one long sequence."""
    wl = Workload("t", HK=2, HV=4, dk=128, dv=128, chunk=64, act="bf16", seed=17, seqlens=(140,),
                  init_state=True, init_conv=True)
    inp = make_inputs(wl)
    T1 = 100
    m = GpuMixer(wl, inp)
    d = m.d
    ys = [m.prefill(x=d["x"][:T1], z=d["z"][:T1], u=d["u"][:T1], b=d["b_logit"][:T1],
                    cu=torch.tensor([0, T1], dtype=torch.int32, device="cuda"))]
    for t in range(T1, 140):
        ys.append(m.decode(d["x"][t:t + 1], d["z"][t:t + 1], d["u"][t:t + 1], d["b_logit"][t:t + 1]))
    ref = oracle_mixer(wl, inp)
    assert rel_max(torch.cat(ys), ref["y"]) <= TOL_BF16
    assert rel_max(m.state, ref["state"]) <= TOL_BF16


def test_deterministic_bitwise():
    wl = Workload("t", HK=2, HV=4, dk=128, dv=128, chunk=64, act="bf16", seed=18, seqlens=(90, 200),
                  init_state=True, init_conv=True)
    inp = make_inputs(wl)
    a, b = GpuMixer(wl, inp), GpuMixer(wl, inp)
    assert torch.equal(a.prefill(), b.prefill())
    assert torch.equal(a.state, b.state)


# ------------------------------------------------------ standalone entry points

def test_standalone_entry_points():
    wl = Workload("t", HK=2, HV=4, dk=64, dv=64, chunk=16, act="bf16", seed=19, seqlens=(40, 9),
                  init_state=True, init_conv=True)
    inp = make_inputs(wl)
    cfg = gdn.make_config(wl.HK, wl.HV, wl.dk, wl.dv, wl.chunk, wl.act, n_slots=2)
    d = {k: dev(v) for k, v in inp.items() if hasattr(v, "to")}
    T = d["x"].shape[0]
    # gate prep
    g = torch.empty((T, wl.HV), device="cuda"); beta = torch.empty_like(g)
    gdn.gdn_gate_prep(cfg, d["u"], d["b_logit"], d["A_log"], d["dt_bias"], g, beta)
    rg, rb = oracle.gates(inp["u"], inp["b_logit"], inp["A_log"], inp["dt_bias"])
    assert rel_max(g, rg) <= 1e-5 and rel_max(beta, rb) <= 1e-5
    # conv prefill (fp32 out) with history
    xa = torch.empty((T, wl.CH), device="cuda")
    conv = d["conv_state"].clone()
    gdn.gdn_conv1d_prefill(cfg, d["x"], d["cu_seqlens"], d["conv_w"], conv, None, xa)
    rxa, rcs = oracle.conv1d_silu(inp["x"], inp["cu_seqlens"], inp["conv_w"], inp["conv_state"])
    assert rel_max(xa, rxa) <= 1e-5
    assert torch.equal(conv.float().cpu(), torch.tensor(rcs, dtype=torch.float32))
    # chunk prefill on the conv output, L2 in the kernel, fp32 o
    o = torch.empty((T, wl.HV * wl.dv), device="cuda")
    st_out = torch.empty_like(d["state"])
    H = wl.HK * wl.dk
    cws = torch.empty(max(gdn.gdn_workspace_size(cfg, T, len(inp["cu_seqlens"]) - 1), 16),
                      dtype=torch.uint8, device="cuda")
    gdn.gdn_chunk_prefill(cfg, xa[:, :H], xa[:, H:2 * H], xa[:, 2 * H:], g, beta, d["cu_seqlens"],
                          d["state"], st_out, None, o, workspace=cws)
    rxn = oracle.l2norm_qk(rxa, wl.HK, wl.dk)
    ro, rst = oracle.delta_rule(rxn, rg, rb, inp["cu_seqlens"], wl.HK, wl.HV, wl.dk, wl.dv,
                                state=inp["state"])
    assert rel_max(o, ro) <= 1e-4 and rel_max(st_out, rst) <= 1e-4
    # gated norm, fp32 and bf16 y
    y = torch.empty_like(o)
    gdn.gdn_gated_rmsnorm(cfg, o, d["z"], d["norm_w"], y)
    ry = oracle.gated_rmsnorm(ro, inp["z"], inp["norm_w"], wl.HV, wl.dv)
    assert rel_max(y, ry) <= TOL_BF16
    # conv step + recurrent decode on one token per sequence
    x1 = d["x"][:2].contiguous()
    conv2 = d["conv_state"].clone()
    xa1 = torch.empty((2, wl.CH), device="cuda")
    gdn.gdn_conv1d_step(cfg, x1, d["conv_w"], conv2, None, xa1)
    rxa1, rcs1 = oracle.conv1d_silu(inp["x"][:2], [0, 1, 2], inp["conv_w"], inp["conv_state"])
    assert rel_max(xa1, rxa1) <= 1e-5
    assert torch.equal(conv2.float().cpu(), torch.tensor(rcs1, dtype=torch.float32))
    st = d["state"].clone()
    o1 = torch.empty((2, wl.HV * wl.dv), device="cuda")
    gdn.gdn_recurrent_decode(cfg, xa1[:, :H], xa1[:, H:2 * H], xa1[:, 2 * H:], g[:2], beta[:2], st,
                             None, o1)
    ro1, rst1 = oracle.delta_rule(oracle.l2norm_qk(rxa1, wl.HK, wl.dk), rg[:2], rb[:2], [0, 1, 2],
                                  wl.HK, wl.HV, wl.dk, wl.dv, state=inp["state"])
    assert rel_max(o1, ro1) <= 1e-4 and rel_max(st, rst1) <= 1e-4


def test_device_error_word_reports_bad_metadata():
    """Malformed cu_seqlens and an out-of-range slot are clamped in the kernels
    (every access stays in bounds) and reported through the error word."""
    wl = Workload("t", HK=2, HV=2, dk=32, dv=32, chunk=16, act="fp32", seed=20, seqlens=(10, 10),
                  init_state=True, init_conv=True)
    inp = make_inputs(wl)
    m = GpuMixer(wl, inp)
    assert gdn.gdn_device_error() == 0
    m.prefill(cu=torch.tensor([0, 15, 5], dtype=torch.int32, device="cuda"))   # not monotone, != T
    code = gdn.gdn_device_error()
    assert code & gdn.DEVERR_CU_SEQLENS
    assert gdn.gdn_device_error() == 0                                        # cleared
    m2 = GpuMixer(wl, inp, state_idx=torch.tensor([0, 7], dtype=torch.int32), n_slots=2)
    m2.prefill()
    assert gdn.gdn_device_error() & gdn.DEVERR_SLOT
