"""bench.py's contract pieces that need no GPU: the reference arm's JSON line (the oracle timed
on the host cores) and the algorithmic counts the roofline fractions divide by."""
import importlib.util
import json
import os
import subprocess
import sys

from gateddeltanet_linear_attention_gb300.inputs import WORKLOADS

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_mod2", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_reference_arm_prints_one_contract_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--steps", "1", "--warmup", "0"], capture_output=True, text=True, timeout=600,
                         cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline",
                "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["unit"] == "tokens/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]
    assert d["config"]["workload"].startswith("prefill_8k")


def test_algorithmic_counts():
    b = _bench()
    # contraction FLOPs of one full chunk of 64 tokens and one v-head at d = 128:
    # 2C^2dk (KK^T) + 2C^2dk (QK^T) + 2C^2dk (W) + 2C^2dv (U) + 2C^2dv (intra O)
    # + 3 * 2C dk dv (W M, Q M, K~^T U') + 2C^3/3 (solve)
    C, d = 64, 128
    per_chunk = 6 * C * C * d + 4 * C * C * d + 6 * C * d * d + 2 * C ** 3 / 3
    assert round(per_chunk) == 11_709_099
    assert b.chunk_flops([64], 64, 128, 128, 1) == per_chunk
    assert abs(b.chunk_flops([8192], 64, 128, 128, 32) - 128 * 32 * per_chunk) <= 1e-9 * 128 * 32 * per_chunk
    # a partial chunk counts at its own length
    L = 20
    part = 6 * L * L * d + 4 * L * L * d + 6 * L * d * d + 2 * L ** 3 / 3
    assert abs(b.chunk_flops([64 + L], 64, 128, 128, 1) - (per_chunk + part)) <= 1e-6
    # step bytes of prefill_8k: x (8192 channels) + z + y (4096 each) in bf16 and g, beta in fp32
    # per token; the fp32 state written once (zero initial state) and the bf16 history written
    wl = WORKLOADS["prefill_8k"]
    per_tok = 8192 * 2 + 2 * 4096 * 2 + 2 * 32 * 4
    assert b.step_hbm_bytes(wl, 8192, 1) == 8192 * per_tok + 32 * 128 * 128 * 4 + 8192 * 3 * 2
