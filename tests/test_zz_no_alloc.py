"""gdn_mixer_prefill_static: the prefill entry point for callers that cannot
allocate device memory (its intermediates live in a fixed scratch array inside
the library).  Checked against gdn_mixer_prefill, which uses a caller
workspace, on two calls in a row; the file sorts last so that a run stopping
at the first failure has already run every other test."""
import pytest
import torch

from gateddeltanet_linear_attention_gb300 import gdn
from gateddeltanet_linear_attention_gb300.inputs import Workload, make_inputs

from gpu_util import TOL_BF16, TOL_FP32, rel_max

pytestmark = pytest.mark.gpu


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


@pytest.mark.parametrize("wl,tol", [
    (Workload("noalloc_bf16", HK=16, HV=32, dk=128, dv=128, chunk=64, act="bf16", seed=21,
              seqlens=(100, 37, 200), init_state=True, init_conv=True), TOL_BF16),
    (Workload("noalloc_fp32", HK=2, HV=4, dk=64, dv=64, chunk=16, act="fp32", seed=22,
              seqlens=(50, 0, 77), init_state=True, init_conv=True), TOL_FP32),
])
def test_static_scratch_matches_workspace_entry_point(wl, tol):
    inp = make_inputs(wl)
    d = {k: v.cuda() for k, v in inp.items() if hasattr(v, "cuda")}
    cfg = gdn.make_config(wl.HK, wl.HV, wl.dk, wl.dv, wl.chunk, wl.act, n_slots=len(wl.seqlens))
    ref = _run(None, wl, d, cfg, static=False)
    for _ in range(2):                      # two calls in a row share the scratch array
        got = _run(None, wl, d, cfg, static=True)
        for g, r in zip(got, ref):
            assert rel_max(g, r.double().cpu().numpy()) <= tol
    assert gdn.gdn_device_error() == 0


def test_static_scratch_rejects_oversize_batch():
    wl = Workload("big", HK=16, HV=32, dk=128, dv=128, chunk=64, act="bf16", seed=23,
                  seqlens=(1,))
    cfg = gdn.make_config(wl.HK, wl.HV, wl.dk, wl.dv, wl.chunk, wl.act, n_slots=1)
    per_token = gdn.gdn_workspace_size(cfg, 1000, 1) / 1000
    T = int((64 << 20) / per_token) + 16       # just past what the fixed scratch holds
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
