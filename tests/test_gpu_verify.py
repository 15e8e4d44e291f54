"""Multi-token verification decode on the GPU against the oracle (hyperflare
core-design, speculative target state: one recurrent checkpoint column per
verification input, continuation from the column of the last accepted one).

gdn_mixer_verify runs k tokens per sequence from a source slot and writes the
state and conv history after every token to its own slot.  Compared with
oracle.mixer_verify (the plain mixer over the k prefixes): y and every
column's state within the bf16 tolerance (1e-4 in fp32 mode), the conv
columns exactly (they are copies of raw inputs), the source slots bit for
bit untouched.  Then: padding lanes, out-of-range columns, and committing a
column followed by ordinary decode steps."""
import numpy as np
import pytest
import torch

import oracle
from gateddeltanet_linear_attention_gb300 import gdn

from gpu_util import TOL_BF16, TOL_FP32, rel_max, report

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    gdn.load()


class Case:
    """Seeded inputs of one verification round: n sequences x k tokens, a pool of `slots`."""

    def __init__(self, n, k, slots, HK=2, HV=4, d=128, act="bf16", seed=0):
        self.n, self.k, self.HK, self.HV, self.d = n, k, HK, HV, d
        self.CH = 2 * HK * d + HV * d
        self.dt = torch.bfloat16 if act == "bf16" else torch.float32
        self.cfg = gdn.make_config(HK, HV, d, d, 64 if d == 128 else 16, act, slots)
        g = torch.Generator().manual_seed(seed)
        r = lambda *s, std=1.0: (torch.randn(*s, generator=g) * std)
        T = n * k
        self.x, self.z = r(T, self.CH).to(self.dt), r(T, HV * d).to(self.dt)
        self.u, self.b = r(T, HV).to(self.dt), r(T, HV).to(self.dt)
        self.cw = r(self.CH, 4, std=0.25).to(self.dt)
        self.A = torch.rand(HV, generator=g) * 2 - 1
        self.dtb = torch.zeros(HV)
        self.nw = torch.ones(d)
        self.state = r(slots, HV, d, d, std=0.02)
        self.conv = r(slots, self.CH, 3).to(self.dt)

    def run(self, src, ckpt, y_dtype=torch.float32):
        dv = lambda t: t.cuda().contiguous()
        self.gs, self.gc = dv(self.state), dv(self.conv)
        y = torch.full((self.n * self.k, self.HV * self.d), 7.0, dtype=y_dtype, device="cuda")
        ws = torch.empty(gdn.gdn_workspace_size(self.cfg, self.n * self.k, self.n), dtype=torch.uint8,
                         device="cuda")
        gdn.gdn_mixer_verify(self.cfg, dv(self.x), dv(self.z), dv(self.u), dv(self.b), dv(self.cw),
                             dv(self.A), dv(self.dtb), dv(self.nw), y, self.gs, self.gc,
                             torch.tensor(ckpt, dtype=torch.int32, device="cuda"), self.k, ws,
                             state_idx=torch.tensor(src, dtype=torch.int32, device="cuda"))
        torch.cuda.synchronize()
        return y

    def oracle(self, src):
        return oracle.mixer_verify(self.x, self.cw, self.u, self.b, self.A, self.dtb, self.z, self.nw,
                                   self.k, self.HK, self.HV, self.d, self.d, self.state, self.conv,
                                   src_idx=src)


def _check(case, src, ckpt, tol, name):
    y = case.run(src, ckpt)
    assert gdn.gdn_device_error() == 0
    ry, rs, rc = case.oracle(src)
    ey = rel_max(y, ry)
    es = max(rel_max(case.gs[ckpt[i]:ckpt[i] + case.k], rs[i]) for i in range(case.n))
    report(name, y=ey, columns=es)
    assert ey <= tol and es <= tol, (ey, es)
    for i in range(case.n):
        got = case.gc[ckpt[i]:ckpt[i] + case.k].float().cpu().numpy()
        assert np.array_equal(got, rc[i])                              # raw inputs: exact
    for s in src:                                                      # sources untouched
        assert torch.equal(case.gs[s].cpu(), case.state[s])
        assert torch.equal(case.gc[s].cpu(), case.conv[s])
    return y


@pytest.mark.parametrize("k", [1, 5, 8])
def test_verify_matches_oracle_bf16(k):
    case = Case(n=3, k=k, slots=3 + 3 * 8, seed=k)
    _check(case, [2, 0, 1], [3 + 8 * i for i in range(3)], TOL_BF16, "verify k=%d" % k)


def test_verify_gqa4_and_fp32_mode():
    case = Case(n=2, k=6, slots=2 + 12, HK=1, HV=4, seed=11)
    _check(case, [1, 0], [2, 8], TOL_BF16, "verify gqa4")
    case = Case(n=2, k=3, slots=2 + 6, HK=2, HV=2, d=32, act="fp32", seed=12)
    _check(case, [0, 1], [2, 5], TOL_FP32, "verify fp32 d=32")


def test_verify_column0_over_source_and_bf16_y():
    """A sequence's own source slot may be its column 0 (read before it is written); bf16 y is
    the rounded fp32 y."""
    case = Case(n=1, k=4, slots=4, seed=14)
    ry, rs, _ = case.oracle([0])
    y = case.run([0], [0])
    assert gdn.gdn_device_error() == 0
    assert rel_max(y, ry) <= TOL_BF16 and rel_max(case.gs[0:4], rs[0]) <= TOL_BF16
    yb = case.run([0], [0], y_dtype=torch.bfloat16)
    assert torch.equal(yb, y.to(torch.bfloat16))


def test_verify_padding_lane_and_rejected_columns():
    case = Case(n=3, k=4, slots=12, seed=15)
    y = case.run([0, -1, 1], [4, 8, 20])       # lane 1 padding; lane 2's columns reach past the pool
    assert gdn.gdn_device_error() == 2
    ry, rs, _ = case.oracle([0, 0, 1])
    assert torch.all(y[4:] == 0)                                       # lanes 1 and 2: zero outputs
    assert rel_max(y[:4], ry[:4]) <= TOL_BF16
    assert torch.equal(case.gs[8:12].cpu(), case.state[8:12])          # padding lane wrote nothing
    assert torch.equal(case.gc[8:12].cpu(), case.conv[8:12])


def test_commit_then_decode_continues_the_accepted_prefix():
    """Verify 5 tokens, accept 3, continue with 2 ordinary decode steps from column 2: the
    outputs equal the oracle over the 3 accepted tokens followed by the 2 new ones."""
    case = Case(n=1, k=5, slots=1 + 5, seed=16)
    y = case.run([0], [1])
    assert gdn.gdn_device_error() == 0
    g = torch.Generator().manual_seed(99)
    nx = (torch.randn(2, case.CH, generator=g)).to(case.dt)
    nz = (torch.randn(2, case.HV * case.d, generator=g)).to(case.dt)
    nu = (torch.randn(2, case.HV, generator=g)).to(case.dt)
    nb = (torch.randn(2, case.HV, generator=g)).to(case.dt)
    commit = torch.tensor([1 + 3 - 1], dtype=torch.int32, device="cuda")
    ws = torch.empty(gdn.gdn_workspace_size(case.cfg, 1, 1), dtype=torch.uint8, device="cuda")
    ys = []
    for t in range(2):
        yt = torch.empty((1, case.HV * case.d), device="cuda")
        gdn.gdn_mixer_decode(case.cfg, nx[t:t + 1].cuda(), nz[t:t + 1].cuda(), nu[t:t + 1].cuda(),
                             nb[t:t + 1].cuda(), case.cw.cuda(), case.A.cuda(), case.dtb.cuda(),
                             case.nw.cuda(), yt, case.gs, case.gc, ws, state_idx=commit)
        ys.append(yt)
    torch.cuda.synchronize()
    assert gdn.gdn_device_error() == 0
    xs = torch.cat([case.x[:3], nx]); zs = torch.cat([case.z[:3], nz])
    us = torch.cat([case.u[:3], nu]); bs = torch.cat([case.b[:3], nb])
    ref = oracle.mixer(xs, case.cw, us, bs, case.A, case.dtb, zs, case.nw, np.array([0, 5], np.int32),
                       case.HK, case.HV, case.d, case.d, state=oracle._f64(case.state[:1]),
                       conv_state=oracle._f64(case.conv[:1]))
    got = torch.cat([y[:3]] + ys)
    assert rel_max(got, ref["y"]) <= TOL_BF16
    assert rel_max(case.gs[3:4], ref["state"]) <= TOL_BF16
    assert np.array_equal(case.gc[3:4].float().cpu().numpy(), ref["conv_state"])
