"""Host-side logic of bench.py that decides reported numbers: the algorithmic work behind every
roofline fraction, and the gating of recorded DRAM traffic on the kernel source it was
measured on.  CPU only."""
import hashlib
import os

import numpy as np

import bench
from fp8_gemm_sigmoid_b300 import synthetic as sy


def test_stage_work_matches_the_layer_closed_forms():
    # Prefill shape: per token, 8 routed rows and the shared expert's row go through
    # [gate; up] (2*H*2I flops each) and down (2*I*H flops each).
    cfg = sy.config("v3_prefill")
    T, H, I, K = cfg["T"], cfg["hidden"], cfg["inter"], cfg["top_k"]
    w = bench.stage_work(cfg)
    per_token = (w["gemm1_swiglu"][1] + w["gemm2_down"][1]) / T
    assert per_token == (K + 1) * (2 * H * 2 * I + 2 * I * H)
    assert abs(per_token / 1e6 - 792.7) < 0.05  # 792.7 MFLOP per token at H=7168, I=2048
    assert w["gemm1_swiglu"][0] == w["gemm2_down"][0] == "tensor"
    # the gate reads x (BF16) and Wg once; the combine reads 9 BF16 rows and writes y per token
    assert w["gate"][1] >= T * H * 2 and w["gate"][1] < T * H * 2 * 1.05
    assert w["combine"][1] >= (K + 1) * T * H * 2 + T * H * 2
    for k in ("gate", "quant", "gate_quant", "permute", "combine"):
        assert w[k][0] == "hbm"
    # fused, x is read once: the two stages' bytes less one read of x
    assert w["gate_quant"][1] == w["gate"][1] + w["quant"][1] - T * H * 2
    # no shared expert: one row per routed slot only
    cfg0 = dict(cfg, has_shared=0)
    assert bench.stage_work(cfg0)["gemm2_down"][1] == T * K * 2 * I * H


def _sha(stage):
    return bench.source_digest(bench.KERNEL_SOURCES[stage])


def test_source_digest_covers_the_included_headers(tmp_path, monkeypatch):
    csrc = tmp_path / "fp8_gemm_sigmoid_b300" / "csrc"
    csrc.mkdir(parents=True)
    (tmp_path / "include").mkdir()
    (csrc / "k.cu").write_text('#include "a.cuh"\n#include <stdio.h>\nkernel\n')
    (csrc / "a.cuh").write_text('#include "../../include/api.h"\n#include "k.cu"\n')
    (tmp_path / "include" / "api.h").write_text("v1\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    d1 = bench.source_digest("k.cu")
    (tmp_path / "include" / "api.h").write_text("v2\n")   # two includes down
    d2 = bench.source_digest("k.cu")
    assert d1 != d2
    whole = hashlib.sha256((csrc / "k.cu").read_bytes() + (csrc / "a.cuh").read_bytes() + b"v2\n")
    assert d2 == whole.hexdigest()   # each file once, in first-inclusion order


def test_measured_traffic_is_reported_only_for_the_measured_source(tmp_path, monkeypatch):
    # a capture on a cut-down case (T=2048, 32 experts: the same rows per expert) scales to the
    # full workload by the tokens processed
    f = tmp_path / "traffic.txt"
    f.write_text("# workload stage sha read write T E\n"
                 "v3_prefill gate %s 1000 24 2048 256\n"
                 "v3_prefill combine %s 7 8 2048 32\n"
                 "v3_prefill quant %s 7 8 2048 64\n"
                 "v3_prefill permute %s 100 28 2048 32\n"
                 "v3_prefill mx/gemm1_swiglu %s 500 12 2048 32\n"
                 % (_sha("gate"), "0" * 64, _sha("quant"), _sha("permute"), _sha("mx/gemm1_swiglu")))
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(f))
    full = sy.config("v3_prefill")
    assert bench.measured_traffic("gate", full)[0] == 1024 * 8       # the gate keeps E, scales by T
    assert bench.measured_traffic("gate", sy.config("v3_prefill", T=2048))[0] == 1024
    assert bench.measured_traffic("gate", sy.config("v3_prefill", T=2048, n_experts=32)) == (None, None)
    assert bench.measured_traffic("permute", full)[0] == 128 * 8      # same rows per expert
    assert bench.measured_traffic("combine", full) == (None, None)   # source changed since
    assert bench.measured_traffic("quant", full) == (None, None)     # another rows-per-expert shape
    assert bench.measured_traffic("gemm1_swiglu", full) == (None, None)   # only the MX kernel captured
    assert bench.measured_traffic("gemm1_swiglu", dict(full, mode="mxfp8"))[0] == 512 * 8
    assert bench.measured_traffic("gate", sy.config("v3_decode")) == (None, None)  # other workload
    assert bench.measured_traffic("bias_update", full) == (None, None)
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(tmp_path / "absent.txt"))
    assert bench.measured_traffic("gate", full) == (None, None)


def test_recorded_traffic_file_is_well_formed():
    with open(bench.TRAFFIC_FILE) as f:
        rows = [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]
    for workload, stage, sha, rd, wr, cap_T, cap_E in rows:
        assert workload in sy.CONFIGS and stage in bench.KERNEL_SOURCES
        assert len(sha) == 64 and int(sha, 16) >= 0
        assert int(rd) > 0 and int(wr) >= 0 and int(cap_T) > 0 and int(cap_E) > 0


def test_gemm_rows_counts_whole_tiles():
    r = bench.gemm_rows([0, 1, 128, 129, 256], T=300, has_shared=1)
    assert r["useful"] == 0 + 1 + 128 + 129 + 256 + 300
    assert r["tile_rows"] == (0 + 1 + 1 + 2 + 2 + 3) * 128
    assert r["tile_efficiency"] == r["useful"] / r["tile_rows"]


def test_tensor_peak_follows_the_clock_regime():
    peaks = dict(bf16=1747.0, bf16_sus=1378.6, hbm=6494.3, src="measured")
    burst = bench.tensor_peak(peaks, {"sm_mhz": 2032.0, "sm_max_mhz": 2032.0, "samples": 40, "reasons": []})
    assert burst == (1747.0 * 2, "burst")
    capped = {"sm_mhz": 1440.0, "sm_max_mhz": 2032.0, "samples": 51, "reasons": ["sw_power_cap"]}
    peak, label = bench.tensor_peak(peaks, capped)
    assert peak == 1378.6 * 2 and label.startswith("sustained")
    # too few samples, or full clock despite the flag, or no record: the burst figure
    assert bench.tensor_peak(peaks, dict(capped, samples=3))[1] == "burst"
    assert bench.tensor_peak(peaks, dict(capped, sm_mhz=2010.0))[1] == "burst"
    assert bench.tensor_peak(peaks, None)[1] == "burst"


def test_gemm_bytes_count_the_hit_experts_once():
    cfg = sy.config("v3_decode")
    T, H, I, K = cfg["T"], cfg["hidden"], cfg["inter"], cfg["top_k"]
    R = T * K + T
    counts = np.zeros(cfg["n_experts"], np.int64)
    counts[[3, 7]] = [T * K - 5, 5]                 # two experts hit, plus the shared one
    b = bench.gemm_bytes(cfg, counts)
    w13 = 3 * (2 * I * H + (2 * I // 128) * (H // 128) * 4)
    assert b["gemm1_swiglu"] == w13 + R * (H + H // 128 * 4) + R * (I + I // 128 * 4)
    w2 = 3 * (H * I + (H // 128) * (I // 128) * 4)
    assert b["gemm2_down"] == w2 + R * (I + I // 128 * 4) + R * H * 2
    # decode with every expert hit streams 11.3 GB of FP8 weights: HBM-bound, not tensor-bound
    full = bench.gemm_bytes(cfg, np.ones(cfg["n_experts"]))
    peaks = dict(bf16=1747.0, bf16_sus=1378.6, hbm=6494.3)
    flops = bench.stage_work(cfg)["gemm1_swiglu"][1]
    assert full["gemm1_swiglu"] / (peaks["hbm"] * 1e9) > flops / (2 * peaks["bf16"] * 1e12)
    prefill = sy.config("v3_prefill")
    pb = bench.gemm_bytes(prefill, np.ones(prefill["n_experts"]))
    assert pb["gemm1_swiglu"] / (peaks["hbm"] * 1e9) < bench.stage_work(prefill)["gemm1_swiglu"][1] / (
        2 * peaks["bf16"] * 1e12)


def test_reference_arm_runs_the_oracle_plan(capsys):
    # the reference arm on a small FP8 layer, on the CPU: one JSON line describing the plan
    import json
    import types
    cfg = sy.config("v3_decode", T=96, hidden=256, inter=128, n_experts=16, n_group=4, topk_group=2, top_k=4)
    args = types.SimpleNamespace(ref_gate_tokens=64, ref_sample=16, steps=2, warmup=1)
    bench.run_reference(args, cfg, 0, 1)
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0 and line["unit"] == "tokens/s"
    assert line["cpu_baseline"]["kind"] == "oracle" and "16-token sample" in line["cpu_baseline"]["sample"]
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["value"] == line["value"]
    bench.run_reference(args, cfg, 1, 2)          # other ranks print nothing
    assert capsys.readouterr().out == ""
