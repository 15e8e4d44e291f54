"""gdn_mixer_prefill_static: the prefill entry point for callers that cannot
allocate device memory (its intermediates live in a fixed scratch array inside
the library).  Checked against gdn_mixer_prefill, which uses a caller
workspace, on two calls in a row: both run the same deterministic kernels on
the same inputs, so the results must be identical.  The file sorts last so
that a run stopping at the first failure has already run every other test."""
import os
import re

import pytest
import torch

from gateddeltanet_linear_attention_gb300 import gdn
from gateddeltanet_linear_attention_gb300.inputs import Workload, make_inputs

pytestmark = pytest.mark.gpu


def _scratch_bytes():
    """GDN_STATIC_SCRATCH_BYTES as include/gdn.h defines it."""
    hdr = open(os.path.join(os.path.dirname(__file__), "..", "include", "gdn.h")).read()
    m = re.search(r"#define\s+GDN_STATIC_SCRATCH_BYTES\s+\((\d+)u\s*<<\s*(\d+)\)", hdr)
    return int(m.group(1)) << int(m.group(2))


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    gdn.load()


def _run(fn, wl, d, cfg, static):
    st = d["state"].clone()
    conv = d["conv_state"].clone()
    T = d["x"].shape[0]
    y = torch.empty((T, wl.HV * wl.dv), device="cuda")
    args = (cfg, d["x"], d["z"], d["u"], d["b_logit"], d["conv_w"], d["A_log"], d["dt_bias"],
            d["norm_w"], d["cu_seqlens"], y)
    if static:
        gdn.gdn_mixer_prefill_static(*args, state_in=st, state_out=st, conv_state=conv)
    else:
        N = d["cu_seqlens"].shape[0] - 1
        ws = torch.empty(gdn.gdn_workspace_size(cfg, T, N), dtype=torch.uint8, device="cuda")
        gdn.gdn_mixer_prefill(*args, state_in=st, state_out=st, conv_state=conv, workspace=ws)
    torch.cuda.synchronize()
    return y, st, conv


@pytest.mark.parametrize("wl", [
    Workload("noalloc_bf16", HK=16, HV=32, dk=128, dv=128, chunk=64, act="bf16", seed=21,
             seqlens=(100, 37, 200), init_state=True, init_conv=True),
    Workload("noalloc_fp32", HK=2, HV=4, dk=64, dv=64, chunk=16, act="fp32", seed=22,
             seqlens=(50, 0, 77), init_state=True, init_conv=True),
])
def test_static_scratch_matches_workspace_entry_point(wl):
    inp = make_inputs(wl)
    d = {k: v.cuda() for k, v in inp.items() if hasattr(v, "cuda")}
    cfg = gdn.make_config(wl.HK, wl.HV, wl.dk, wl.dv, wl.chunk, wl.act, n_slots=len(wl.seqlens))
    ref = _run(None, wl, d, cfg, static=False)
    for _ in range(2):                      # two calls in a row share the scratch array
        got = _run(None, wl, d, cfg, static=True)
        for g, r in zip(got, ref):
            assert torch.equal(g, r)
    assert gdn.gdn_device_error() == 0


def test_static_scratch_rejects_oversize_batch():
    wl = Workload("big", HK=16, HV=32, dk=128, dv=128, chunk=64, act="bf16", seed=23,
                  seqlens=(1,))
    cfg = gdn.make_config(wl.HK, wl.HV, wl.dk, wl.dv, wl.chunk, wl.act, n_slots=1)
    limit = _scratch_bytes()
    lo, hi = 1, 1 << 20                        # the first T whose workspace exceeds the scratch
    while hi - lo > 1:
        mid = (lo + hi) // 2
        if gdn.gdn_workspace_size(cfg, mid, 1) > limit:
            hi = mid
        else:
            lo = mid
    T = hi + 16                                # (at d=128 in bf16 the prefill part dominates)
    x = torch.zeros((T, wl.CH), dtype=torch.bfloat16, device="cuda")
    z = torch.zeros((T, wl.HV * wl.dv), dtype=torch.bfloat16, device="cuda")
    ub = torch.zeros((T, wl.HV), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros((wl.CH, 4), dtype=torch.bfloat16, device="cuda")
    hv = torch.zeros(wl.HV, device="cuda")
    nw = torch.ones(wl.dv, device="cuda")
    cu = torch.tensor([0, T], dtype=torch.int32, device="cuda")
    y = torch.empty((T, wl.HV * wl.dv), device="cuda")
    with pytest.raises(gdn.GDNError) as ei:
        gdn.gdn_mixer_prefill_static(cfg, x, z, ub, ub, w, hv, hv, nw, cu, y)
    assert ei.value.status == 3          # GDN_ERR_WORKSPACE: the batch needs more scratch
