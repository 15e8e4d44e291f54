"""The device-side timeout path, exercised without a GPU fault.

Every wait of a kernel on another part of itself (an mbarrier a copy or a peer
arrives on) is bounded: it gives up after the configured limit, records
GDN_DEVERR_TIMEOUT, writes no state and returns (hyperflare core-design:
unsupported conditions end in a typed failure, never a hang).  Here the limit
is shortened to 20 ms and a launch is told to drop one operand copy, so a wait
really runs out.  The kernel must return by itself, the error word must hold
the timeout bit, the state it would have written must be untouched, and the
next normal call must match the oracle."""
import numpy as np
import pytest
import torch

from gateddeltanet_linear_attention_gb300 import gdn
from gateddeltanet_linear_attention_gb300.inputs import Workload, make_inputs

from gpu_util import TOL_BF16, GpuMixer, oracle_mixer, rel_max, report

pytestmark = pytest.mark.gpu

SHORT_NS = 20_000_000


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    gdn.load()
    yield
    gdn.gdn_debug_set_wait()          # defaults back, whatever happened


def test_decode_state_wait_runs_out_then_recovers():
    wl = Workload("timeout_decode", HK=2, HV=4, dk=128, dv=128, chunk=64, act="bf16", seed=51,
                  init_state=True, init_conv=True, decode_steps=2, n_decode=8)
    inp = make_inputs(wl)
    m = GpuMixer(wl, inp)
    before = m.state.clone()
    conv_before = m.conv.clone()
    gdn.gdn_debug_set_wait(SHORT_NS, 1)
    try:
        y = m.decode(inp["dec_x"][0].cuda(), inp["dec_z"][0].cuda(), inp["dec_u"][0].cuda(),
                     inp["dec_b_logit"][0].cuda())
        code = gdn.gdn_device_error()
    finally:
        gdn.gdn_debug_set_wait()
    assert code & gdn.DEVERR_TIMEOUT
    # the streaming CTA that lost its copy (unit 0: sequence 0, v-heads 0 and 1) wrote no state
    # and zero outputs; every other head was updated
    assert torch.equal(m.state[0, :2], before[0, :2])
    assert torch.all(y[0, :2 * wl.dv] == 0)
    assert not torch.equal(m.state[1:], before[1:])
    # the next normal call, from the original state, matches the oracle
    m.state.copy_(before); m.conv.copy_(conv_before)
    y = m.decode(inp["dec_x"][1].cuda(), inp["dec_z"][1].cuda(), inp["dec_u"][1].cuda(),
                 inp["dec_b_logit"][1].cuda())
    torch.cuda.synchronize()
    assert gdn.gdn_device_error() == 0
    cu = np.arange(wl.n_decode + 1, dtype=np.int32)
    ref = oracle_mixer(wl, inp, x=inp["dec_x"][1], u=inp["dec_u"][1], b=inp["dec_b_logit"][1],
                       z=inp["dec_z"][1], cu=cu)
    ey, es = rel_max(y, ref["y"]), rel_max(m.state, ref["state"])
    report("decode after a timeout", y=ey, state=es)
    assert ey <= TOL_BF16 and es <= TOL_BF16


def test_chain_operand_wait_runs_out_then_recovers():
    wl = Workload("timeout_prefill", HK=2, HV=4, dk=128, dv=128, chunk=64, act="bf16", seed=52,
                  seqlens=(200, 77), init_state=True, init_conv=True)
    inp = make_inputs(wl)
    m = GpuMixer(wl, inp, y_dtype=torch.float32)
    before = m.state.clone()
    gdn.gdn_debug_set_wait(SHORT_NS, 2)
    try:
        m.prefill()
        code = gdn.gdn_device_error()
    finally:
        gdn.gdn_debug_set_wait()
    assert code & gdn.DEVERR_TIMEOUT
    assert torch.equal(m.state, before)            # no chain CTA stored a state
    # a normal call on fresh buffers matches the oracle
    m = GpuMixer(wl, inp, y_dtype=torch.float32)
    y = m.prefill()
    torch.cuda.synchronize()
    assert gdn.gdn_device_error() == 0
    ref = oracle_mixer(wl, inp)
    ey, es = rel_max(y, ref["y"]), rel_max(m.state, ref["state"])
    report("prefill after a timeout", y=ey, state=es)
    assert ey <= TOL_BF16 and es <= TOL_BF16
