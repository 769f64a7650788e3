"""Benchmark of the MoE layer forward (gate -> quantise -> permute -> grouped FP8 GEMM with
SwiGLU -> grouped FP8 GEMM down-projection -> combine with the shared expert) on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config v3_prefill] [--impl ours|reference]

Prints ONE JSON line (rank 0).  A step is one whole layer forward over T tokens of the named
workload (default: the DeepSeek-V3-shaped prefill layer, T=16384).  Inputs are seeded
synthetic tensors with the workload's shapes and distributions, resident in HBM before
timing; the 11.3 GB of FP8 expert weights are far larger than L2, so no flush is needed.
With N > 1 (torchrun), every rank runs its own T tokens (independent replicas, weak
scaling; the layer has no cross-token exchange) and the slowest rank's time counts.
"""
import argparse
import datetime
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from fp8_gemm_sigmoid_b300 import moe, replicas, synthetic as sy  # noqa: E402

PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "dram_traffic.txt")
KERNEL_SOURCES = {"gemm1_swiglu": "gemm_tc.cu", "gemm2_down": "gemm_tc.cu", "gate": "gate.cu", "gate_quant": "gate.cu",
                  "quant": "quant.cu", "permute": "permute.cu", "combine": "combine.cu",
                  "mx/gemm1_swiglu": "gemm_mx.cu", "mx/gemm2_down": "gemm_mx.cu"}
FP8_PER_BF16 = 2.0  # nominal dense FP8 / BF16 tensor rate (4.5 / 2.25 PFLOP/s)
STAGED_SECONDS = 2.5  # the per-stage pass runs at least this long (>= 20 clock samples)

# kernels each entry point launches in the FP8 layer (memsets excluded); summed into
# gpu_launches.  moe_permute: chunk histogram, scan, positions, row gather, scale gather.
# Each grouped GEMM is one persistent kernel (its tile schedule is built in shared memory).
LAUNCHES = {"moe_gate": 1, "moe_quant_1x128": 1, "moe_gate_quant": 1, "moe_permute": 5,
            "moe_grouped_gemm_fp8/swiglu": 1, "moe_grouped_gemm_fp8/store": 1,
            "moe_combine": 1, "moe_bias_update": 1}


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=40)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--config", default="v3_prefill", choices=sorted(sy.CONFIGS))
    p.add_argument("--mode", default=None, choices=["fp8", "mxfp8"],
                   help="quantisation mode of the timed layer (default: the workload's, FP32 scales)")
    p.add_argument("--no-mxfp8", action="store_true",
                   help="skip the secondary measurement of the power-of-two (MXFP8) mode")
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--cpu-sample", type=int, default=512,
                   help="tokens of the seeded sample on which the oracle's expert FFNs are timed")
    p.add_argument("--ref-gate-tokens", type=int, default=2048,
                   help="reference arm: tokens per step through the oracle's gate")
    p.add_argument("--ref-sample", type=int, default=64,
                   help="reference arm: tokens per step through the oracle's expert FFNs")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--staged-seconds", type=float, default=STAGED_SECONDS,
                   help="minimum length of the per-stage pass (0: exactly --steps steps, for profiling)")
    # smaller variants of the workload for profiler captures (same per-expert row count
    # when T*top_k/experts is kept)
    p.add_argument("--T", type=int, default=None)
    p.add_argument("--experts", type=int, default=None)
    p.add_argument("--groups", type=int, default=None)
    p.add_argument("--topk-group", type=int, default=None)
    # one stage alone (a profiler's target with a small device footprint)
    p.add_argument("--only", choices=["gate", "gate_quant"], default=None)
    return p.parse_args()


def load_peaks():
    try:
        with open(PEAKS_FILE) as f:
            P = json.load(f)
        return dict(hbm=P["hbm_gbs"], bf16=P["bf16_tflops"], bf16_sus=P["bf16_tflops_sustained"],
                    src="measured")
    except (OSError, KeyError, ValueError):
        return dict(hbm=6400.0, bf16=1800.0, bf16_sus=1400.0, src="fallback")


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons, started before the timed regions;
    stats(t0, t1) summarises the samples whose timestamps fall inside one region."""
    Q = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    PERIOD_MS = 50

    def __init__(self, index):
        self.index = index
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        self.rows = None
        try:
            self.p = subprocess.Popen(["nvidia-smi", "-i", str(index), "--query-gpu=" + self.Q,
                                       "--format=csv,noheader,nounits", "-lms", str(self.PERIOD_MS)],
                                      stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.p = None
        # wait (bounded) for the first sample, so that the timed regions are covered
        t_end = time.time() + 10
        while self.p is not None and time.time() < t_end:
            if os.path.getsize(self.f.name) > 0:
                break
            time.sleep(0.05)

    @staticmethod
    def now():
        return datetime.datetime.now()

    def stop(self):
        if self.p is None:
            return
        self.p.terminate()
        self.p.wait()
        self.f.flush()
        rows = []
        with open(self.f.name) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 10:
                    continue
                try:
                    ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f")
                except ValueError:
                    continue
                rows.append([ts] + parts[1:])
        os.unlink(self.f.name)
        self.rows = rows

    def stats(self, t0, t1):
        if not self.rows:
            return None
        rows = [r for r in self.rows if t0 <= r[0] <= t1]
        if not rows:  # a region shorter than one period: the samples around it
            before = [r for r in self.rows if r[0] < t0][-1:]
            after = [r for r in self.rows if r[0] > t1][:1]
            rows = before + after
        if not rows:
            return None
        num = lambda v: v.replace(".", "").isdigit()  # noqa: E731
        sm = [float(r[2]) for r in rows if num(r[2])]
        pw = [float(r[4]) for r in rows if num(r[4])]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            for n, v in zip(names, r[6:10]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": float(rows[0][3]) if num(rows[0][3]) else None,
                "power_w_max": max(pw) if pw else None,
                "samples": len(rows), "reasons": sorted(reasons)}


class Layer:
    """Device-resident inputs, FP8 weights, outputs, staged intermediates and workspace."""

    def __init__(self, cfg, dev, keep_bf16=True, inp=None, extra_modes=(), q=None):
        """inp: inputs to share with another Layer; q: its FP8 weights, already quantised;
        extra_modes: other quantisation modes whose FP8 weights are made before the BF16
        weights are dropped (self.extra_q[mode])."""
        self.cfg = cfg
        T, H, I, E, K = cfg["T"], cfg["hidden"], cfg["inter"], cfg["n_experts"], cfg["top_k"]
        S = int(cfg["has_shared"])
        self.mx = cfg["mode"] == "mxfp8"
        self.inp = inp if inp is not None else sy.make_inputs(cfg, dev)
        self.q = q if q is not None else moe.quantize_weights(self.inp["W13"], self.inp["W2"], pow2=self.mx)
        self.extra_q = {m: moe.quantize_weights(self.inp["W13"], self.inp["W2"], pow2=(m == "mxfp8"))
                        for m in extra_modes}
        if not keep_bf16 and inp is None:  # the BF16 expert weights only feed the CPU oracle
            del self.inp["W13"], self.inp["W2"]
            torch.cuda.empty_cache()
        self.x = self.inp["x"].view(torch.uint16)
        self.weights = dict(Wg=self.inp["Wg"].view(torch.uint16), **self.q)
        self.bias = self.inp["bias"].clone()
        self.out = moe.empty_outputs(cfg, T, dev)
        self.y = self.out["y"].view(torch.uint16)
        self.ws = moe.workspace(cfg, T, dev)
        R = T * K + T * S
        self.R = R
        u8, f32, i32 = torch.uint8, torch.float32, torch.int32
        self.xq = torch.empty(T, H, dtype=u8, device=dev)
        self.xs = torch.empty(T, H // 128, dtype=f32, device=dev)
        self.offs = torch.empty(E + 2, dtype=i32, device=dev)
        self.perm_tok = torch.empty(R, dtype=i32, device=dev)
        self.row_of = torch.empty(T, K, dtype=i32, device=dev)
        self.aq = torch.empty(R, H, dtype=u8, device=dev)
        self.as_ = torch.empty(H // 128, R, dtype=f32, device=dev)  # K-block-major
        self.hq = torch.empty(R, I, dtype=u8, device=dev)
        self.hs = torch.empty(I // 128, R, dtype=f32, device=dev)  # K-block-major
        self.yexp = torch.empty(R, H, dtype=torch.bfloat16, device=dev)
        # FP8 modes: from MOE_GATE_QUANT_MIN_TOKENS tokens up the gate quantises x in the same
        # pass when its tensor-core kernel takes the shape (moe_forward then launches no separate
        # quantiser); the staged pass does the same
        self.fused = False
        if cfg["T"] >= moe.MOE_GATE_QUANT_MIN_TOKENS:
            try:
                o = self.out
                moe.moe_gate_quant(cfg, self.x, self.weights["Wg"], self.bias, o["topk_idx"], o["topk_w"],
                                   o["counts"], self.xq, self.xs)
                self.fused = True
            except moe.MoEError as e:
                if e.status != moe.MOE_ERR_UNSUPPORTED:
                    raise
        self.stages = (["gate_quant"] if self.fused else ["gate", "quant"]) + Layer.STAGES[2:]

    def forward(self, world=1):
        """One layer step.  Under N > 1 token replicas the top-1 bias update runs after an
        all-reduce of the histogram, so every rank updates from the whole batch's load."""
        o = self.out
        replicated = world > 1 and self.cfg["update_bias"]
        moe.moe_forward(self.cfg, self.x, self.weights, self.bias,
                        0 if replicated else self.cfg["update_bias"], self.y,
                        o["topk_idx"], o["topk_w"], o["counts"], self.ws)
        if replicated:
            replicas.global_bias_update(self.cfg, o["counts"], self.cfg["T"], self.bias,
                                        lambda c, Tg, cnt, b: moe.moe_bias_update(c, Tg, cnt, b),
                                        T_global=world * self.cfg["T"])

    STAGES = ["gate", "quant", "permute", "gemm1_swiglu", "gemm2_down", "combine", "bias_update"]

    def staged(self, ev, world=1):
        """The same layer through the individual entry points, an event before the first stage
        and after each of self.stages (len(self.stages) + 1 events)."""
        c, o = self.cfg, self.out
        T, H, I, E = c["T"], c["hidden"], c["inter"], c["n_experts"]
        G = E + int(c["has_shared"])
        ev = iter(ev)
        next(ev).record()
        if self.fused:
            moe.moe_gate_quant(c, self.x, self.weights["Wg"], self.bias, o["topk_idx"], o["topk_w"], o["counts"],
                               self.xq, self.xs)
            next(ev).record()
        else:
            moe.moe_gate(c, self.x, self.weights["Wg"], self.bias, o["topk_idx"], o["topk_w"], o["counts"])
            next(ev).record()
            if self.mx:
                moe.moe_quant_1x128_pow2(self.x, self.xq, self.xs)
            else:
                moe.moe_quant_1x128(self.x, self.xq, self.xs)
            next(ev).record()
        moe.moe_permute(c, T, o["topk_idx"], o["counts"], self.xq, self.xs, self.offs, self.perm_tok,
                        self.row_of, self.aq, self.as_, self.ws)
        next(ev).record()
        if self.mx:
            moe.moe_grouped_gemm_mxfp8(G, self.offs, self.R, 2 * I, H, self.aq, self.as_, self.q["W13"],
                                       self.q["W13_s"], moe.MOE_EPI_SWIGLU_QUANT, self.hq, self.hs)
        else:
            moe.moe_grouped_gemm_fp8(G, self.offs, self.R, 2 * I, H, self.aq, self.as_, self.q["W13"],
                                     self.q["W13_s"], moe.MOE_EPI_SWIGLU_QUANT, self.hq, self.hs, self.ws)
        next(ev).record()
        if self.mx:
            moe.moe_grouped_gemm_mxfp8(G, self.offs, self.R, H, I, self.hq, self.hs, self.q["W2"],
                                       self.q["W2_s"], moe.MOE_EPI_STORE, self.yexp, None)
        else:
            moe.moe_grouped_gemm_fp8(G, self.offs, self.R, H, I, self.hq, self.hs, self.q["W2"],
                                     self.q["W2_s"], moe.MOE_EPI_STORE, self.yexp, None, self.ws)
        next(ev).record()
        ysh = self.yexp[T * c["top_k"]:] if c["has_shared"] else None
        moe.moe_combine(c, T, self.yexp, self.row_of, o["topk_w"], ysh, self.y)
        next(ev).record()
        if c["update_bias"]:
            if world > 1:  # token replicas: the update from the whole batch's histogram
                replicas.global_bias_update(c, o["counts"], T, self.bias,
                                            lambda cc, Tg, cnt, b: moe.moe_bias_update(cc, Tg, cnt, b),
                                            T_global=world * T)
            else:
                moe.moe_bias_update(c, T, o["counts"], self.bias)
        next(ev).record()

    def launches_per_step(self):
        first = ("moe_gate_quant",) if self.fused else ("moe_gate", "moe_quant_1x128")
        n = sum(LAUNCHES[k] for k in first + ("moe_permute", "moe_grouped_gemm_fp8/swiglu",
                                              "moe_grouped_gemm_fp8/store", "moe_combine"))
        return n + (LAUNCHES["moe_bias_update"] if self.cfg["update_bias"] else 0)


def stage_work(cfg):
    """Algorithmic work of each stage: FLOPs for the GEMMs, bytes for the rest."""
    T, H, I, E, K = cfg["T"], cfg["hidden"], cfg["inter"], cfg["n_experts"], cfg["top_k"]
    S = int(cfg["has_shared"])
    R = T * K + T * S
    return {
        "gate": ("hbm", T * H * 2 + E * H * 2 + T * K * 8 + E * 4),
        "quant": ("hbm", T * H * 2 + T * H + T * (H // 128) * 4),
        # the gate with the quantisation fused in: x read once, the codes and scales written
        "gate_quant": ("hbm", T * H * 2 + E * H * 2 + T * K * 8 + E * 4 + T * H + T * (H // 128) * 4),
        "permute": ("hbm", T * K * 4 * 3 + R * (H + H // 128 * 4) + T * (H + H // 128 * 4)),
        "gemm1_swiglu": ("tensor", 2 * R * H * 2 * I),
        "gemm2_down": ("tensor", 2 * R * I * H),
        "combine": ("hbm", R * H * 2 + T * H * 2 + T * K * 8),
        "bias_update": ("hbm", E * 12),
    }


def gemm_bytes(cfg, counts):
    """Algorithmic HBM bytes of each grouped GEMM: the FP8 weights and scales of every expert
    that received a row (and of the shared expert), the A rows and scales read, and the output
    written.  At small T (decode) these, not the FLOPs, bound the GEMMs."""
    T, H, I, K = cfg["T"], cfg["hidden"], cfg["inter"], cfg["top_k"]
    S = int(cfg["has_shared"])
    R = T * K + T * S
    n_w = int((np.asarray(counts) > 0).sum()) + S
    w13 = n_w * (2 * I * H + (2 * I // 128) * (H // 128) * 4)
    w2 = n_w * (H * I + (H // 128) * (I // 128) * 4)
    return {"gemm1_swiglu": w13 + R * (H + H // 128 * 4) + R * (I + I // 128 * 4),
            "gemm2_down": w2 + R * (I + I // 128 * 4) + R * H * 2}


def source_digest(name):
    """SHA-256 over a kernel source file of csrc/ and every file it includes with quotes,
    transitively, in first-inclusion order: any edit to the code the kernel is built from
    changes it."""
    import hashlib
    import re
    h = hashlib.sha256()
    seen = []

    def walk(path):
        path = os.path.normpath(path)
        if path in seen:
            return
        seen.append(path)
        with open(path, "rb") as f:
            text = f.read()
        h.update(text)
        for inc in re.findall(rb'^\s*#\s*include\s+"([^"]+)"', text, re.M):
            walk(os.path.join(os.path.dirname(path), inc.decode()))

    walk(os.path.join(ROOT, "fp8_gemm_sigmoid_b300", "csrc", name))
    return h.hexdigest()


def measured_traffic(stage, cfg):
    """DRAM bytes (read + write) of one launch of the stage's kernel on cfg's workload, from the
    ncu counters recorded in profiles/dram_traffic.txt, or (None, None) when no capture of the
    kernel's current source exists.  A capture is taken on a cut-down case of the workload's
    shape (fewer tokens and experts, the same rows per expert); its bytes scale to cfg's
    workload by the tokens processed.  Each line of the file records source_digest() of the
    kernel's source at capture time, and a line only counts while that digest is unchanged.
    The gate's bytes (the tokens, their T x K outputs and the [E, H] gate weight) scale by the
    tokens at the same E, so its capture keeps the experts instead.
    Power-of-two (MXFP8) stages are recorded as mx/<stage>."""
    if cfg.get("mode") == "mxfp8" and stage.startswith("gemm"):
        stage = "mx/" + stage
    src = KERNEL_SOURCES.get(stage)
    if src is None or not os.path.exists(TRAFFIC_FILE):
        return None, None
    sha = source_digest(src)
    with open(TRAFFIC_FILE) as f:
        for line in f:
            parts = line.split()
            if line.startswith("#") or len(parts) < 7:
                continue
            workload, st, digest, rd, wr, cap_T, cap_E = parts[:7]
            same_shape = int(cap_E) * cfg["T"] == int(cap_T) * cfg["n_experts"]
            if stage in ("gate", "gate_quant"):  # x, the T x K outputs, the [E, H] gate weight: same E, any T
                same_shape = int(cap_E) == cfg["n_experts"]
            if workload == cfg["name"] and st == stage and digest == sha and same_shape:
                scale = cfg["T"] / int(cap_T)
                return int(round((int(rd) + int(wr)) * scale)), "ncu capture at T=%s E=%s scaled by tokens x%.3g" % (cap_T, cap_E, scale)
    return None, None


def tensor_peak(peaks, clk):
    """FP8 tensor peak for a kernel timed in a region with clock record clk: the measured
    BF16 burst figure x 2, or the sustained (seconds-long, power-capped) figure x 2 when the
    region's median SM clock sat below 95 % of its maximum with sw_power_cap active -- the
    regime the sustained figure was measured in.  Returns (peak TFLOP/s, regime label)."""
    if clk and clk.get("samples", 0) >= 5 and "sw_power_cap" in clk.get("reasons", ()) and \
            clk.get("sm_mhz") and clk.get("sm_max_mhz") and clk["sm_mhz"] < 0.95 * clk["sm_max_mhz"]:
        return peaks["bf16_sus"] * FP8_PER_BF16, "sustained (power-capped region, %.0f of %.0f MHz)" % (
            clk["sm_mhz"], clk["sm_max_mhz"])
    return peaks["bf16"] * FP8_PER_BF16, "burst"


def barrier_sync(dist_on):
    if dist_on:
        torch.distributed.barrier()
    if torch.cuda.is_available():
        torch.cuda.synchronize()


def max_over_ranks(v, dist_on):
    """The slowest rank's value (replica timing); a CUDA tensor under NCCL, a CPU one under gloo."""
    if not dist_on:
        return v
    dev = "cuda" if torch.distributed.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(tokens_per_rank, steps, ms_per_rank, dist_on):
    """Whole-job tokens/s of independent replicas: every rank's tokens over the slowest rank's
    time."""
    world = torch.distributed.get_world_size() if dist_on else 1
    ms = max_over_ranks(ms_per_rank, dist_on)
    return world * tokens_per_rank * steps / (ms / 1e3), ms


class OracleLayer:
    """The CPU oracle on the workload's inputs (host copies), with the expert weights it needs
    quantised on the oracle side beforehand: quantisation of the weights is an offline step on
    both sides, so no timed region contains it."""

    def __init__(self, cfg, inp):
        """inp: the workload's inputs as synthetic.make_inputs draws them (BF16 expert weights
        included)."""
        import numpy as np
        import oracle
        self.np, self.oracle, self.cfg = np, oracle, cfg
        self.pow2 = cfg["mode"] == "mxfp8"
        self.ocfg = dict(cfg, mode="fp8_pow2") if self.pow2 else cfg  # the oracle's name of the mode
        self.x = inp["x"].view(torch.uint16).cpu().numpy()
        self.Wg = inp["Wg"].view(torch.uint16).cpu().numpy()
        self.bias = inp["bias"].cpu().numpy()
        self.W13, self.W2 = inp["W13"], inp["W2"]
        self.cache = {}

    def qweights(self, ids):
        np = self.np
        miss = [int(e) for e in ids if int(e) not in self.cache]
        if miss:
            idx = torch.tensor(miss, device=self.W13.device)
            w13 = self.W13.index_select(0, idx).view(torch.uint16).cpu().numpy()
            w2 = self.W2.index_select(0, idx).view(torch.uint16).cpu().numpy()
            q = self.oracle.quantize_weights(w13, w2, pow2=self.pow2)
            for j, e in enumerate(miss):
                self.cache[e] = tuple(a[j:j + 1] for a in q)
        return tuple(np.concatenate([self.cache[int(e)][i] for e in ids]) for i in range(4))

    def gate(self, tokens):
        c = self.cfg
        return self.oracle.gate(self.x[tokens], self.Wg, self.bias, c["n_group"], c["topk_group"], c["top_k"],
                                c["routed_scaling_factor"])

    def prepare(self, g, sample):
        """Quantise (untimed) the experts that `sample`'s tokens of routing `g` reach."""
        ids = self.np.unique(self.np.concatenate([g["topk_idx"][sample].ravel(), [self.cfg["n_experts"]]]))
        self.qweights(ids)

    def timed(self, gate_tokens, sample):
        """One pass of the plan: gate and permutation over `gate_tokens` (a contiguous range of
        the batch), then the expert FFNs and the combine for `sample` (indices into that range).
        Returns (gate seconds, expert seconds)."""
        c = self.cfg
        t0 = time.perf_counter()
        g = self.gate(gate_tokens)
        self.oracle.permute(g["topk_idx"], c["n_experts"], int(c["has_shared"]))
        t1 = time.perf_counter()
        self.prepare(g, sample)
        t2 = time.perf_counter()
        self.oracle.experts_and_combine(self.ocfg, self.x[gate_tokens], g, sample, None, None, qweights=self.qweights)
        t3 = time.perf_counter()
        return t1 - t0, t3 - t2


def cpu_baseline(cfg, layer, n_sample):
    """The oracle, as it stands, on the host cores: the gate and the permutation over all T
    tokens, then the expert FFNs and the combine on a seeded sample of n_sample tokens.  Every
    output row depends only on its own token, so the expert part extrapolates per token:
    tokens/s = T / (gate time + expert time * T / n_sample)."""
    T = cfg["T"]
    ol = OracleLayer(cfg, layer.inp)
    sample = sy.sample_tokens(T, n_sample, seed=2).numpy()
    g = ol.gate(slice(0, T))
    ol.prepare(g, sample)  # weights quantised outside the timed passes
    t_gate, t_exp = ol.timed(slice(0, T), sample)
    n = len(sample)
    value = T / (t_gate + t_exp * T / n)
    return {"value": value, "unit": "tokens/s", "cores": ol.oracle.num_threads(), "kind": "oracle",
            "sample": "gate + permutation over all %d tokens (%.2f s), expert FFNs + combine on a seeded "
                      "%d-token sample (%.2f s), extrapolated per token to %d tokens"
                      % (T, t_gate, n, t_exp, T)}


def run_reference(args, cfg, rank, world):
    """The reference arm: the CPU oracle timed on the host cores, rank 0 only.  Each step runs
    the cpu_baseline plan on a bounded slice of the batch (gate + permutation over a run of
    ref_gate_tokens tokens, expert FFNs + combine on a seeded sample of ref_sample of them) and
    the per-token times extrapolate to the workload's T, as cpu_baseline's do."""
    if rank != 0:
        return
    import numpy as np
    dev = "cuda:0" if torch.cuda.is_available() else "cpu"
    if dev != "cpu":
        torch.cuda.set_device(0)
    # the workload's inputs, drawn as for the library's arm; nothing of the library runs here
    ol = OracleLayer(cfg, sy.make_inputs(cfg, dev))
    T = cfg["T"]
    n_gate = min(args.ref_gate_tokens, T)
    n_exp = min(args.ref_sample, n_gate)

    def step(i):
        start = (i * 7919 * n_gate) % max(1, T - n_gate + 1)
        sample = np.sort(np.random.default_rng(1000 + i).choice(n_gate, n_exp, replace=False))
        rng = slice(start, start + n_gate)
        ol.prepare(ol.gate(rng), sample)
        return ol.timed(rng, sample)

    for i in range(args.warmup):
        step(i)
    per_token = 0.0
    tot = 0.0
    for i in range(args.steps):
        tg, te = step(args.warmup + i)
        per_token += tg / n_gate + te / n_exp
        tot += tg + te
    val = args.steps / per_token
    line = {
        "impl": "reference", "metric": metric_name(cfg), "value": val,
        "unit": "tokens/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": tot / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_dict(cfg, 1),
        "cpu_baseline": {"value": val, "unit": "tokens/s", "cores": ol.oracle.num_threads(), "kind": "oracle",
                         "sample": "per step: gate + permutation over %d consecutive tokens of the %s batch, "
                                   "expert FFNs + combine on a seeded %d-token sample of them; per-token "
                                   "times extrapolated to the batch (the plan of cpu_baseline on a smaller "
                                   "slice)" % (n_gate, cfg["name"], n_exp)},
        "e2e": {"value": val, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def gemm_rows(counts, T, has_shared, bm=128):
    """Rows the grouped GEMMs compute: the algorithmic rows and the rows of whole bm-row tiles."""
    import numpy as np
    c = np.asarray(counts, np.int64)
    useful = int(c.sum()) + (T if has_shared else 0)
    tiles = int(np.sum((c + bm - 1) // bm)) + ((T + bm - 1) // bm if has_shared else 0)
    return {"useful": useful, "tile_rows": tiles * bm, "tile_efficiency": useful / max(1, tiles * bm)}


def metric_name(cfg):
    return "MoE layer tokens/s and grouped-GEMM TFLOPS (%% of FP8 peak) at T=%d, 1 B300" % cfg["T"]


def config_dict(cfg, world):
    return {"workload": cfg["name"], "T": cfg["T"], "hidden": cfg["hidden"], "inter": cfg["inter"],
            "n_experts": cfg["n_experts"], "top_k": cfg["top_k"], "shared": cfg["has_shared"],
            "l2": "inputs larger than L2 (11.3 GB of FP8 expert weights per step)",
            "parallelism": "replicas x%d" % world}


def run_only(args, cfg):
    """moe_gate (or moe_gate_quant) alone on the workload's tokens: K timed calls after W warm-up
    calls."""
    torch.cuda.set_device(0)
    T = cfg["T"]
    inp = sy.make_inputs(cfg, "cuda", weights=False)
    out = moe.empty_outputs(cfg, T)
    fp8 = cfg["mode"] == "fp8"
    x = inp["x"].view(torch.uint16) if fp8 else inp["x"]
    Wg = inp["Wg"].view(torch.uint16) if fp8 else inp["Wg"]
    call = lambda: moe.moe_gate(cfg, x, Wg, inp["bias"], out["topk_idx"], out["topk_w"], out["counts"])  # noqa: E731
    if args.only == "gate_quant":
        xq = torch.empty(T, cfg["hidden"], dtype=torch.uint8, device="cuda")
        xs = torch.empty(T, cfg["hidden"] // 128, dtype=torch.float32, device="cuda")
        call = lambda: moe.moe_gate_quant(cfg, x, Wg, inp["bias"], out["topk_idx"], out["topk_w"],  # noqa: E731
                                          out["counts"], xq, xs)
    for _ in range(max(args.warmup, 3)):
        call()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(args.steps):
        call()
    b.record()
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / args.steps
    nbytes = stage_work(cfg)[args.only][1]
    print(json.dumps({"stage": args.only, "workload": cfg["name"], "T": T, "us_per_call": ms * 1e3,
                      "GB/s": nbytes / ms / 1e6, "steps": args.steps}), flush=True)


def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    over = {k: v for k, v in (("T", args.T), ("n_experts", args.experts), ("n_group", args.groups),
                              ("topk_group", args.topk_group)) if v is not None}
    if args.mode is not None:
        over["mode"] = args.mode
    cfg = sy.config(args.config, **over)
    if args.only:
        return run_only(args, cfg)
    if args.impl == "reference":
        return run_reference(args, cfg, rank, world)
    dist_on = world > 1
    if dist_on:
        torch.distributed.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = "cuda:%d" % local
    peaks = load_peaks()
    T = cfg["T"]
    want_cpu = rank == 0 and world == 1 and not args.no_cpu_baseline
    want_mx = cfg["mode"] == "fp8" and not args.no_mxfp8
    layer = Layer(cfg, dev, keep_bf16=want_cpu, extra_modes=("mxfp8",) if want_mx else ())
    stream = torch.cuda.current_stream()

    # warm-up (W whole-layer steps through moe_forward and through the staged calls)
    for _ in range(max(args.warmup, 3)):
        layer.forward(world)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(len(layer.stages) + 1)]
    for _ in range(2):
        layer.staged(ev, world)
    barrier_sync(dist_on)

    # timed region 1: K steps of moe_forward (the headline)
    clocks = Clocks(local)
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier_sync(dist_on)
    r1 = [clocks.now()]
    start.record(stream)
    for _ in range(args.steps):
        layer.forward(world)
    stop.record(stream)
    barrier_sync(dist_on)
    r1.append(clocks.now())
    value, ms = replica_throughput(T, args.steps, start.elapsed_time(stop), dist_on)
    assert moe.moe_device_error() == 0

    # timed region 2: the staged entry points with an event after every stage, repeated for
    # at least STAGED_SECONDS so that the clock record holds enough samples (events for every
    # step up front and one synchronize at the end, so that the host's enqueueing never leaves
    # the GPU idle between stages)
    step_s = ms / args.steps / 1e3
    n_staged = max(args.steps, min(2000, int(args.staged_seconds / max(step_s, 1e-6)) + 1)
                   if args.staged_seconds > 0 else args.steps)
    stage_ms = {s: 0.0 for s in layer.stages}
    barrier_sync(dist_on)
    all_evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(layer.stages) + 1)] for _ in range(n_staged)]
    r2 = [clocks.now()]
    for evs in all_evs:
        layer.staged(evs, world)
    barrier_sync(dist_on)
    r2.append(clocks.now())
    for evs in all_evs:
        for i, s in enumerate(layer.stages):
            stage_ms[s] += evs[i].elapsed_time(evs[i + 1]) / n_staged
    counts = layer.out["counts"].cpu().numpy()

    # end to end through the host-buffer entry points (moe_pipeline_submit): every step
    # uploads its tokens from pinned host memory and downloads y, the routing and the
    # histogram; consecutive steps' copies overlap each other's compute.  Host-clock timing
    # from the first submit to the last step's outputs in host memory.
    e2e = None
    if not args.no_e2e:
        o = layer.out
        pin = lambda t: torch.empty(t.shape, dtype=t.dtype).pin_memory()  # noqa: E731
        x_host = pin(layer.x)
        x_host.copy_(layer.x)
        y_host, idx_host, w_host, c_host = pin(layer.y), pin(o["topk_idx"]), pin(o["topk_w"]), pin(o["counts"])
        pl = moe.MoEPipeline(cfg, T, stream=stream)

        def e2e_step():
            pl.submit(x_host, layer.weights, layer.bias, cfg["update_bias"], y_host, idx_host, w_host, c_host)

        for _ in range(2):
            e2e_step()
        pl.wait()
        barrier_sync(dist_on)
        t0 = time.perf_counter()
        for _ in range(args.steps):
            e2e_step()
        pl.wait()
        e2e_s = time.perf_counter() - t0
        barrier_sync(dist_on)
        pl.close()
        e2e_ms = max_over_ranks(e2e_s * 1e3, dist_on)
        h2d = x_host.numel() * x_host.element_size()
        d2h = sum(t.numel() * t.element_size() for t in (y_host, idx_host, w_host, c_host))
        e2e = {"value": world * T * args.steps / (e2e_ms / 1e3), "unit": "tokens/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "api": "moe_pipeline_submit (pinned host buffers)"}
        del pl
        torch.cuda.empty_cache()
    # the LogFMT-8 codec on the combine payload (the routed expert rows, BF16): encode and
    # decode timed apart from the layer step, each K calls between events
    logfmt = None
    if cfg["mode"] == "fp8":
        payload = layer.yexp[:T * cfg["top_k"]].view(torch.uint16)
        rows_l, cols_l = payload.shape
        codes = torch.empty(rows_l, cols_l, dtype=torch.uint8, device=dev)
        lmin = torch.empty(rows_l, cols_l // 128, dtype=torch.float32, device=dev)
        lstep = torch.empty_like(lmin)
        back = torch.empty_like(payload)
        logfmt = {"n_bits": 8, "rows": rows_l, "cols": cols_l}
        for name, fn, nbytes in (
                ("encode", lambda: moe.moe_logfmt_encode(8, payload, codes, lmin, lstep),
                 rows_l * cols_l * 3 + lmin.numel() * 8),
                ("decode", lambda: moe.moe_logfmt_decode(8, codes, lmin, lstep, back),
                 rows_l * cols_l * 3 + lmin.numel() * 8)):
            for _ in range(3):
                fn()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for _ in range(args.steps):
                fn()
            b.record(stream)
            torch.cuda.synchronize()
            t_ms = a.elapsed_time(b) / args.steps
            logfmt[name] = {"ms": t_ms, "GB/s": nbytes / t_ms / 1e6, "frac_hbm": nbytes / t_ms / 1e6 / peaks["hbm"]}
        del codes, lmin, lstep, back
    # the same layer in power-of-two (MXFP8) mode: tensor cores apply the scales themselves
    mxfp8 = None
    if want_mx:
        cfg_mx = dict(cfg, mode="mxfp8")
        lmx = Layer(cfg_mx, dev, keep_bf16=False, inp=layer.inp, q=layer.extra_q.pop("mxfp8"))
        for _ in range(3):
            lmx.forward(world)
        barrier_sync(dist_on)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(args.steps):
            lmx.forward(world)
        b.record(stream)
        barrier_sync(dist_on)
        mx_value, mx_ms = replica_throughput(T, args.steps, a.elapsed_time(b), dist_on)
        evs_mx = [[torch.cuda.Event(enable_timing=True) for _ in range(len(lmx.stages) + 1)] for _ in range(args.steps)]
        for evs in evs_mx:
            lmx.staged(evs, world)
        barrier_sync(dist_on)
        assert moe.moe_device_error() == 0
        k1 = lmx.stages.index("gemm1_swiglu")
        g1 = sum(evs[k1].elapsed_time(evs[k1 + 1]) for evs in evs_mx) / args.steps
        g2 = sum(evs[k1 + 1].elapsed_time(evs[k1 + 2]) for evs in evs_mx) / args.steps
        w_mx = stage_work(cfg)
        mxfp8 = {"value": mx_value, "unit": "tokens/s", "ms_per_step": mx_ms / args.steps,
                 "gemm1_swiglu": {"ms": g1, "TFLOP/s": w_mx["gemm1_swiglu"][1] / g1 / 1e9,
                                  "frac_fp8_peak": w_mx["gemm1_swiglu"][1] / g1 / 1e9 / (peaks["bf16"] * FP8_PER_BF16)},
                 "gemm2_down": {"ms": g2, "TFLOP/s": w_mx["gemm2_down"][1] / g2 / 1e9,
                                "frac_fp8_peak": w_mx["gemm2_down"][1] / g2 / 1e9 / (peaks["bf16"] * FP8_PER_BF16)},
                 "dtype": "fp8-e4m3, power-of-two 1x128 / 128x128 scales applied by the tensor cores"}
        del lmx
        torch.cuda.empty_cache()
    clocks.stop()
    clk = clocks.stats(*r1)
    stage_clk = clocks.stats(*r2)

    work = stage_work(cfg)
    # the grouped GEMMs' denominator: the BF16 figure of the regime their timed region ran in
    # (burst, or sustained when the clocks show the power cap) times the nominal FP8:BF16 ratio
    fp8_peak, regime = tensor_peak(peaks, stage_clk)
    gbytes = gemm_bytes(cfg, counts)
    stages = {}
    for s in layer.stages:
        if s == "bias_update" and not cfg["update_bias"]:
            continue
        kind, amount = work[s]
        t = stage_ms[s] / 1e3
        if kind == "tensor":
            # a GEMM is bound by its FLOPs or by its bytes, whichever takes longer at peak
            ach = amount / t / 1e12 if t > 0 else None
            gbs = gbytes[s] / t / 1e9 if t > 0 else None
            bound = "tensor" if amount / (fp8_peak * 1e12) >= gbytes[s] / (peaks["hbm"] * 1e9) else "hbm"
            stages[s] = {"ms": stage_ms[s], "bound": bound, "TFLOP/s": ach,
                         "frac_fp8_peak": ach / fp8_peak if ach else None,
                         "GB/s": gbs, "frac_hbm": gbs / peaks["hbm"] if gbs else None}
        else:
            ach = amount / t / 1e9 if t > 0 else None
            stages[s] = {"ms": stage_ms[s], "GB/s": ach, "frac_hbm": ach / peaks["hbm"] if ach else None}
    dom = max(stages, key=lambda s: stages[s]["ms"])
    kind, amount = work[dom]
    if kind == "tensor" and stages[dom]["bound"] == "hbm":
        kind, amount = "hbm", gbytes[dom]
    dom_t = stage_ms[dom] / 1e3
    if kind == "tensor":
        roof = {"kernel": dom, "bound": "tensor", "achieved": amount / dom_t / 1e12, "peak": fp8_peak,
                "unit": "TFLOP/s",
                "peak_source": "%s bf16 %s x %.0f (nominal FP8:BF16), of %s" % (
                    peaks["src"], regime, FP8_PER_BF16, peaks["src"]),
                "frac_of_burst": amount / dom_t / 1e12 / (peaks["bf16"] * FP8_PER_BF16)}
    else:
        roof = {"kernel": dom, "bound": "hbm", "achieved": amount / dom_t / 1e9, "peak": peaks["hbm"],
                "unit": "GB/s", "peak_source": "%s copy bandwidth, of %s" % (peaks["src"], peaks["src"])}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["traffic"], roof["traffic_source"] = measured_traffic(dom, cfg)
    roof["algorithmic"] = amount
    roof["sm_mhz"] = stage_clk["sm_mhz"] if stage_clk else None
    gemm_ms = stage_ms["gemm1_swiglu"] + stage_ms["gemm2_down"]
    gemm_tflops = (work["gemm1_swiglu"][1] + work["gemm2_down"][1]) / (gemm_ms / 1e3) / 1e12

    cpu = None
    if want_cpu:
        cpu = cpu_baseline(cfg, layer, min(args.cpu_sample, T))

    line = {
        "metric": metric_name(cfg),
        "value": value,
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms / args.steps,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": ("fp8-e4m3 (FP32 accumulation), bf16 activations" if cfg["mode"] == "fp8" else
                  "fp8-e4m3, power-of-two scales applied by the tensor cores, bf16 activations"),
        "data": "synthetic",
        "config": config_dict(cfg, world),
        "grouped_gemm": {"ms": gemm_ms, "TFLOP/s": gemm_tflops, "frac_fp8_peak": gemm_tflops / fp8_peak,
                         "rows": gemm_rows(counts, T, cfg["has_shared"])},
        "stages": stages,
        "staged_steps": n_staged,
        "logfmt": logfmt,
        "mxfp8": mxfp8,
        "roofline": roof,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": layer.launches_per_step() * args.steps,
        "clocks": clk,
        "stage_clocks": stage_clk,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist_on:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
