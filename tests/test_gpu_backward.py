"""Backward of the gated delta rule core on the GPU against the oracle
(hyperflare core-design, training plan: the GDN core backward from retained
chunk-boundary states).

gdn_chunk_states writes the state before every chunk; it is compared with the
oracle's forward over each prefix.  gdn_chunk_backward turns d_o (and
d_state_out) into dq, dk, dv, dg, dbeta and d_state_in; compared with
oracle.delta_rule_backward (pinned against central differences of the
forward) element by element, max|delta| / RMS(oracle) <= 1e-4 (the GPU path is
fp32 arithmetic throughout).  Every case runs the backward both ways: with the
per-token p and w that gdn_chunk_states retains, and without them (the walk
recomputes them).  Cases: nonzero initial states, one and three
chunks, a partial last chunk, varlen batches with an empty sequence and a
padding lane, GQA 1/2/4, head dims 32/64/128, chunks of 16 and 64, bf16 and
fp32 inputs."""
import numpy as np
import pytest
import torch

import oracle
from gateddeltanet_linear_attention_gb300 import gdn

from gpu_util import rel_max, report

pytestmark = pytest.mark.gpu
TOL = 1e-4


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    gdn.load()


def _unit(x):
    return x / x.norm(dim=-1, keepdim=True)


class Batch:
    def __init__(self, lens, HK, HV, d, chunk, dtype=torch.float32, slots=None, seed=0, init_state=True):
        self.lens, self.HK, self.HV, self.d, self.C = list(lens), HK, HV, d, chunk
        T = sum(lens)
        self.T, self.N = T, len(lens)
        self.slots = slots if slots is not None else list(range(self.N))
        n_slots = max(self.slots) + 1
        g = torch.Generator().manual_seed(seed)
        rn = lambda *s: torch.randn(*s, generator=g)
        self.q = _unit(rn(T, HK, d)).reshape(T, HK * d).to(dtype)
        self.k = _unit(rn(T, HK, d)).reshape(T, HK * d).to(dtype)
        self.v = rn(T, HV * d).to(dtype)
        self.gl = -torch.nn.functional.softplus(rn(T, HV)) * 0.5
        self.beta = torch.sigmoid(rn(T, HV))
        self.S0 = rn(n_slots, HV, d, d) * 0.05 if init_state else None
        self.d_o = rn(T, HV * d)
        self.dS = rn(n_slots, HV, d, d) * 0.1
        self.cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32)
        self.cfg = gdn.make_config(HK, HV, d, d, chunk, "bf16" if dtype == torch.bfloat16 else "fp32",
                                   n_slots)
        self.n_slots = n_slots

    def xa(self):
        return np.concatenate([oracle._f64(self.q), oracle._f64(self.k), oracle._f64(self.v)], axis=1)

    def gpu_states(self, retain=False):
        nb = gdn.chunk_count(self.lens, self.C)
        bnd = torch.full((max(nb, 1), self.HV, self.d, self.d), float("nan"), device="cuda")
        # (NaN where a padding lane's tokens are: nothing may read them)
        pw = torch.full((max(self.T, 1), self.HV, 2, self.d), float("nan"), device="cuda") if retain else None
        ws = torch.empty(gdn.gdn_backward_workspace_size(self.cfg, self.T, self.N), dtype=torch.uint8,
                         device="cuda")
        gdn.gdn_chunk_states(self.cfg, self.k.cuda(), self.v.cuda(), self.gl.cuda(), self.beta.cuda(),
                             self.cu.cuda(), bnd, ws,
                             state_in=None if self.S0 is None else self.S0.cuda(),
                             state_idx=torch.tensor(self.slots, dtype=torch.int32, device="cuda"),
                             token_pw=pw)
        torch.cuda.synchronize()
        return bnd, ws, pw

    def gpu_backward(self, with_dS=True, with_dS0=True, retain=False):
        bnd, ws, pw = self.gpu_states(retain)
        T, HK, HV, d = self.T, self.HK, self.HV, self.d
        dq = torch.full((T, HK * d), float("nan"), device="cuda"); dk = torch.full_like(dq, float("nan"))
        dv = torch.full((T, HV * d), float("nan"), device="cuda")
        dg = torch.full((T, HV), float("nan"), device="cuda"); db = torch.full_like(dg, float("nan"))
        dS0 = torch.zeros((self.n_slots, HV, d, d), device="cuda") if with_dS0 else None
        gdn.gdn_chunk_backward(self.cfg, self.q.cuda(), self.k.cuda(), self.v.cuda(), self.gl.cuda(),
                               self.beta.cuda(), self.cu.cuda(), bnd, self.d_o.cuda(), dq, dk, dv, dg,
                               db, ws, d_state_out=self.dS.cuda() if with_dS else None,
                               d_state_in=dS0,
                               state_idx=torch.tensor(self.slots, dtype=torch.int32, device="cuda"),
                               token_pw=pw)
        torch.cuda.synchronize()
        return dq, dk, dv, dg, db, dS0

    def oracle_backward(self, with_dS=True):
        S0 = None if self.S0 is None else oracle._f64(self.S0)
        if S0 is None:
            S0 = np.zeros((self.n_slots, self.HV, self.d, self.d))
        return oracle.delta_rule_backward(self.xa(), self.gl, self.beta, self.cu.numpy(), self.HK, self.HV,
                                          self.d, self.d, self.d_o, state=S0, slot_idx=self.slots,
                                          d_state=self.dS if with_dS else None)


def _check_backward(b, name, with_dS=True):
    """Both forms of the walk (recomputed and retained p, w) against one oracle result."""
    dxa, rg, rb, rS0 = b.oracle_backward(with_dS=with_dS)
    HKd = b.HK * b.d
    for retain in (False, True):
        dq, dk, dv, dg, db, dS0 = b.gpu_backward(with_dS=with_dS, retain=retain)
        assert gdn.gdn_device_error() == 0
        errs = dict(dq=rel_max(dq, dxa[:, :HKd]), dk=rel_max(dk, dxa[:, HKd:2 * HKd]),
                    dv=rel_max(dv, dxa[:, 2 * HKd:]), dg=rel_max(dg, rg), dbeta=rel_max(db, rb),
                    dS0=rel_max(dS0, rS0))
        report(name + (" (retained p, w)" if retain else ""), **errs)
        for key, e in errs.items():
            assert e <= TOL, (retain, key, e)


@pytest.mark.parametrize("lens,chunk", [((64,), 64), ((192,), 64), ((16,), 16), ((48,), 16)])
def test_backward_one_and_three_chunks(lens, chunk):
    b = Batch(lens, HK=2, HV=4, d=128 if chunk == 64 else 64, chunk=chunk, seed=len(lens) + lens[0])
    _check_backward(b, "bwd %s C=%d" % (lens, chunk))


def test_chunk_states_match_oracle_prefixes():
    b = Batch((150, 0, 70), HK=1, HV=2, d=64, chunk=64, slots=[2, 0, 1], seed=3)
    bnd, _, pw = b.gpu_states(retain=True)
    assert gdn.gdn_device_error() == 0
    idx = 0
    worst = 0.0
    for n, L in enumerate(b.lens):
        s0 = int(b.cu[n])
        for c in range((L + 63) // 64):
            t = s0 + 64 * c
            _, st = oracle.delta_rule(b.xa()[s0:t], b.gl[s0:t], b.beta[s0:t], np.array([0, t - s0], np.int32),
                                      b.HK, b.HV, b.d, b.d, state=oracle._f64(b.S0)[b.slots[n]:b.slots[n] + 1])
            worst = max(worst, rel_max(bnd[idx], st[0]))
            idx += 1
    assert idx == gdn.chunk_count(b.lens, 64)
    # the retained rows of every 5th token and each sequence's last: p = M^T k with M the
    # oracle's state before the token (the prefix before it), w = beta (v - a p)
    xa, d, grp = b.xa(), b.d, b.HV // b.HK
    worst_p = worst_w = 0.0
    for n, L in enumerate(b.lens):
        s0 = int(b.cu[n])
        for t in sorted(set(list(range(s0, s0 + L, 5)) + ([s0 + L - 1] if L else []))):
            _, st = oracle.delta_rule(xa[s0:t], b.gl[s0:t], b.beta[s0:t], np.array([0, t - s0], np.int32),
                                      b.HK, b.HV, d, d, state=oracle._f64(b.S0)[b.slots[n]:b.slots[n] + 1])
            for h in range(b.HV):
                kv = xa[t, b.HK * d + (h // grp) * d:b.HK * d + (h // grp + 1) * d]
                vv = xa[t, 2 * b.HK * d + h * d:2 * b.HK * d + (h + 1) * d]
                p = st[0, h].T @ kv
                w = float(b.beta[t, h]) * (vv - np.exp(float(b.gl[t, h])) * p)
                worst_p = max(worst_p, rel_max(pw[t, h, 0], p))
                worst_w = max(worst_w, rel_max(pw[t, h, 1], w))
    report("chunk states", bnd=worst, p=worst_p, w=worst_w)
    assert worst <= TOL and worst_p <= TOL and worst_w <= TOL


def test_backward_varlen_gqa_padding_and_partial_chunks():
    b = Batch((70, 0, 33, 130), HK=2, HV=4, d=128, chunk=64, slots=[3, 1, -1, 0], seed=9)
    _check_backward(b, "bwd varlen+padding")
    pad = slice(70, 103)                                            # the padding lane's tokens
    for retain in (False, True):
        dq, dk, dv, dg, db, _ = b.gpu_backward(retain=retain)
        assert torch.all(dv[pad] == 0) and torch.all(dg[pad] == 0) and torch.all(dq[pad] == 0)


@pytest.mark.parametrize("HK,HV,d,chunk", [(1, 4, 32, 16), (4, 4, 64, 16), (2, 4, 128, 64)])
def test_backward_shapes_and_no_final_state_term(HK, HV, d, chunk):
    b = Batch((3 * chunk + 5,), HK=HK, HV=HV, d=d, chunk=chunk, seed=HK * 100 + d, init_state=False)
    _check_backward(b, "bwd HK=%d HV=%d d=%d" % (HK, HV, d), with_dS=False)


def test_backward_bf16_inputs():
    b = Batch((100, 60), HK=2, HV=4, d=128, chunk=64, dtype=torch.bfloat16, seed=77)
    _check_backward(b, "bwd bf16 inputs")


def test_backward_at_the_benchmarked_length():
    """8,192 tokens (the length bench.py times), two q/k heads and their four v-heads: every
    chunk's workspace slab of the full-length walk is compared through the gradients."""
    b = Batch((8192,), HK=2, HV=4, d=128, chunk=64, seed=8192)
    _check_backward(b, "bwd 8192 tokens")
