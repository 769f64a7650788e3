"""bench.py's output contract on a cut-down prefill layer: one JSON line with the keys, types and
relations the benchmark promises (metric, value, roofline with its peak source and traffic,
the end-to-end figure with its copy volumes, the launch count, the clock record), for the
library's arm and for the reference arm."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SMALL = ["--T", "2048", "--experts", "32", "--groups", "8", "--topk-group", "4", "--steps", "3", "--warmup", "3",
         "--staged-seconds", "0.2", "--cpu-sample", "16"]


def _run(args):
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py")] + args, cwd=ROOT, capture_output=True,
                         text=True, timeout=900)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, out.stdout[-2000:]
    return json.loads(lines[0])


def test_bench_line_has_the_contract_keys():
    d = _run(SMALL)
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "roofline", "cpu_baseline", "e2e",
              "gpu_launches", "clocks"):
        assert k in d, k
    assert d["unit"] == "tokens/s" and d["value"] > 0 and d["n_gpus"] == 1 and d["steps"] == 3
    assert d["higher_is_better"] is True and d["scaling"] == "weak" and d["data"] == "synthetic"
    assert d["config"]["workload"] == "v3_prefill" and d["config"]["T"] == 2048
    # value is the tokens of the timed steps over their time
    assert abs(d["value"] - 2048 / (d["ms_per_step"] / 1e3)) <= 1e-6 * d["value"]
    r = d["roofline"]
    assert r["bound"] in ("tensor", "hbm") and r["unit"] in ("TFLOP/s", "GB/s")
    assert abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-9 and 0 < r["frac"] < 1.5
    assert "of measured" in r["peak_source"] or "of fallback" in r["peak_source"]
    assert "traffic" in r
    e = d["e2e"]
    assert e["unit"] == "tokens/s" and e["value"] > 0
    assert e["h2d_bytes_per_step"] == 2048 * 7168 * 2            # the tokens, BF16
    assert e["d2h_bytes_per_step"] >= 2048 * 7168 * 2            # y, BF16, plus the routing
    c = d["cpu_baseline"]
    assert c["kind"] == "oracle" and c["value"] > 0 and c["cores"] >= 1 and "16-token sample" in c["sample"]
    # below MOE_GATE_QUANT_MIN_TOKENS the gate and the quantiser run apart: 10 launches per step
    assert d["gpu_launches"] == 10 * 3
    assert "sm_mhz" in d["clocks"] and "reasons" in d["clocks"]


def test_reference_arm_line():
    d = _run(["--impl", "reference", "--T", "2048", "--experts", "32", "--groups", "8", "--topk-group", "4",
              "--steps", "1", "--warmup", "1", "--ref-gate-tokens", "256", "--ref-sample", "8"])
    assert d["impl"] == "reference" and d["value"] > 0 and d["unit"] == "tokens/s"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
