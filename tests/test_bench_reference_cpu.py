"""The benchmark's reference arm on CPU: every config prints one JSON line that keeps the
bench contract (metric, unit, direction, the oracle as cpu_baseline, a zero-copy e2e entry).

The reference arm times the oracle on the host cores, so it runs here without a GPU; the
budget is cut to a second so that the whole file stays fast.
"""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CONFIGS = {
    "long_draft": ("kv_hbm_gbs", "GB/s"),
    "global_verify": ("kv_hbm_gbs", "GB/s"),
    "accept_verify": ("logits_hbm_gbs", "GB/s"),
    "project_prefill": ("projection_tflops", "TFLOP/s"),
    "conv_block": ("conv_hbm_gbs", "GB/s"),
    "selector_walk": ("selector_gather_gbs", "GB/s"),
}


@pytest.mark.parametrize("config", sorted(CONFIGS))
def test_reference_arm_prints_one_contract_line(config):
    cmd = [sys.executable, "bench.py", "--impl", "reference", "--config", config, "--steps", "1", "--warmup", "0",
           "--ref-budget", "1"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    rec = json.loads(lines[0])
    metric, unit = CONFIGS[config]
    assert rec["impl"] == "reference" and rec["metric"] == metric and rec["unit"] == unit
    assert rec["higher_is_better"] is True and rec["n_gpus"] == 1 and rec["data"] == "synthetic"
    assert rec["value"] > 0 and rec["ms_per_step"] > 0
    assert rec["cpu_baseline"]["kind"] == "oracle" and rec["cpu_baseline"]["value"] == rec["value"]
    assert rec["cpu_baseline"]["cores"] >= 1 and rec["cpu_baseline"]["sample"]
    assert rec["e2e"] == {"value": rec["value"], "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert "workload" in rec["config"]
