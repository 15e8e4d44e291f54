"""Slot maintenance on the GPU (hyperflare core-design, "State operations":
snapshot, restore, initialise and reset as indirect copies over device slot
indices; restored continuation must repeat direct continuation exactly).

gdn_state_copy is compared with the oracle's definition bit for bit (fp32
states and bf16 histories viewed as raw bits), over copies, resets, inactive
lanes, out-of-range indices and one shared pool; then a prefill is
snapshotted, decoded, restored and decoded again, and the two continuations
must agree bit for bit."""
import numpy as np
import pytest
import torch

import oracle
from gateddeltanet_linear_attention_gb300 import gdn
from gateddeltanet_linear_attention_gb300.inputs import Workload, make_inputs

from gpu_util import GpuMixer

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    gdn.load()


def _bits(t):
    """Raw bits of a device tensor as a numpy integer array (exact comparisons)."""
    t = t.detach().cpu().contiguous()
    return t.view(torch.int32 if t.element_size() == 4 else torch.int16).numpy()


def _pools(rng_seed, slots, HK=2, HV=4, d=128):
    CH = 2 * HK * d + HV * d          # the layout _cfg() describes
    g = torch.Generator().manual_seed(rng_seed)
    st = torch.randn((slots, HV, d, d), generator=g)
    cs = torch.randn((slots, CH, 3), generator=g).to(torch.bfloat16)
    return st.cuda(), cs.cuda()


def _cfg(HK=2, HV=4, d=128, slots=8):
    return gdn.make_config(HK, HV, d, d, 64, "bf16", slots)


@pytest.mark.parametrize("pairs", [
    [(3, 0), (-1, 2), (5, -1), (0, 5)],                       # copy, reset, inactive, copy
    [(i, 7 - i) for i in range(4)],                            # a permutation into another pool
    [(-1, i) for i in range(8)],                               # initialise the whole pool
    [],                                                        # no pairs
])
def test_state_copy_matches_oracle_bitwise(pairs):
    c = _cfg()
    ss, sc = _pools(1, 6)
    ds, dc = _pools(2, 8)
    src_idx = torch.tensor([p[0] for p in pairs], dtype=torch.int32, device="cuda")
    dst_idx = torch.tensor([p[1] for p in pairs], dtype=torch.int32, device="cuda")
    exp_s, exp_c, exp_err = oracle.state_copy(_bits(ss), _bits(sc), _bits(ds), _bits(dc),
                                              src_idx.cpu().numpy(), dst_idx.cpu().numpy())
    gdn.gdn_state_copy(c, ss, sc, ds, dc, src_idx, dst_idx)
    torch.cuda.synchronize()
    assert gdn.gdn_device_error() == (2 if exp_err else 0)
    assert np.array_equal(_bits(ds), exp_s)
    assert np.array_equal(_bits(dc), exp_c)


def test_state_copy_out_of_range_is_reported_and_skipped():
    c = _cfg()
    ss, sc = _pools(3, 4)
    ds, dc = _pools(4, 4)
    src_idx = torch.tensor([9, 1, 0], dtype=torch.int32, device="cuda")    # 9: past the source pool
    dst_idx = torch.tensor([0, 6, 3], dtype=torch.int32, device="cuda")    # 6: past the destination
    exp_s, exp_c, exp_err = oracle.state_copy(_bits(ss), _bits(sc), _bits(ds), _bits(dc),
                                              src_idx.cpu().numpy(), dst_idx.cpu().numpy())
    gdn.gdn_state_copy(c, ss, sc, ds, dc, src_idx, dst_idx)
    torch.cuda.synchronize()
    assert exp_err and gdn.gdn_device_error() == 2
    assert gdn.gdn_device_error() == 0                                    # read and cleared
    assert np.array_equal(_bits(ds), exp_s) and np.array_equal(_bits(dc), exp_c)


def test_state_copy_one_pool_states_only_and_history_only():
    """Live rows and snapshot rows in one pool; a NULL part is left alone."""
    c = _cfg()
    st, cs = _pools(5, 8)
    before_cs = _bits(cs).copy()
    src_idx = torch.tensor([0, 1, 2], dtype=torch.int32, device="cuda")
    dst_idx = torch.tensor([4, 5, 6], dtype=torch.int32, device="cuda")
    exp_s, _, _ = oracle.state_copy(_bits(st), None, _bits(st), None, [0, 1, 2], [4, 5, 6])
    gdn.gdn_state_copy(c, st, None, st, None, src_idx, dst_idx)          # states only
    torch.cuda.synchronize()
    assert gdn.gdn_device_error() == 0
    assert np.array_equal(_bits(st), exp_s) and np.array_equal(_bits(cs), before_cs)
    _, exp_c, _ = oracle.state_copy(None, _bits(cs), None, _bits(cs), [3, -1], [7, 0])
    gdn.gdn_state_copy(c, None, cs, None, cs, torch.tensor([3, -1], dtype=torch.int32, device="cuda"),
                       torch.tensor([7, 0], dtype=torch.int32, device="cuda"))  # histories only
    torch.cuda.synchronize()
    assert gdn.gdn_device_error() == 0
    assert np.array_equal(_bits(cs), exp_c) and np.array_equal(_bits(st), exp_s)


def test_snapshot_restore_repeats_continuation_bitwise():
    """Prefill into live slots 0..2, snapshot to 3..5, decode 4 steps, restore, decode the same
    4 steps: outputs, states and histories of the two continuations agree bit for bit, and the
    snapshot rows are untouched by the decode."""
    wl = Workload("t", HK=2, HV=4, dk=128, dv=128, chunk=64, act="bf16", seed=31, seqlens=(70, 5, 130),
                  init_state=True, init_conv=True)
    inp = make_inputs(wl)
    m = GpuMixer(wl, inp, n_slots=6, state_idx=torch.tensor([0, 1, 2], dtype=torch.int32))
    m.state = torch.cat([m.d["state"], torch.zeros_like(m.d["state"])]).contiguous()
    m.conv = torch.cat([m.d["conv_state"], torch.zeros_like(m.d["conv_state"])]).contiguous()
    m.prefill()
    live = torch.tensor([0, 1, 2], dtype=torch.int32, device="cuda")
    snap = torch.tensor([3, 4, 5], dtype=torch.int32, device="cuda")
    gdn.gdn_state_copy(m.cfg, m.state, m.conv, m.state, m.conv, live, snap)     # snapshot
    snap_bits = (_bits(m.state[3:]).copy(), _bits(m.conv[3:]).copy())
    g = torch.Generator().manual_seed(77)
    steps = [(torch.randn((3, wl.CH), generator=g).to(torch.bfloat16).cuda(),
              torch.randn((3, wl.HV * wl.dv), generator=g).to(torch.bfloat16).cuda(),
              torch.randn((3, wl.HV), generator=g).to(torch.bfloat16).cuda(),
              torch.randn((3, wl.HV), generator=g).to(torch.bfloat16).cuda()) for _ in range(4)]

    def run():
        ys = [m.decode(*s).clone() for s in steps]
        return ys, _bits(m.state[:3]).copy(), _bits(m.conv[:3]).copy()

    ya, sa, ca = run()
    assert np.array_equal(_bits(m.state[3:]), snap_bits[0])
    assert np.array_equal(_bits(m.conv[3:]), snap_bits[1])
    gdn.gdn_state_copy(m.cfg, m.state, m.conv, m.state, m.conv, snap, live)     # restore
    yb, sb, cb = run()
    torch.cuda.synchronize()
    assert gdn.gdn_device_error() == 0
    for a, b in zip(ya, yb):
        assert torch.equal(a, b)
    assert np.array_equal(sa, sb) and np.array_equal(ca, cb)
