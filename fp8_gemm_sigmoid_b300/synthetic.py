"""Seeded synthetic inputs for the MoE layer workloads.

This module holds no arithmetic of the method: it only draws the layer's inputs (tokens,
gate weight, selection bias, expert weights) from the stated distributions, so the CUDA
path and the CPU oracle can be fed the very same bits.  Large tensors are drawn on the
requested device with a seeded torch generator; small ones (bias, expert permutation) are
always drawn on the CPU.  BF16 tensors are rounded from FP32 draws.

Workloads (the layer shapes of DeepSeek-V3: hidden 7168, 256 routed experts of FFN width
2048 in 8 groups, 4 groups kept, 8 experts per token, 1 shared expert):
  tiny_fp32   T=64, hidden 256, 16 experts / 4 groups, keep 2, top-2, inter 128,
              FP32 throughout; x~N(0,1), weights~N(0,0.02), bias~U(-0.1,0.1)
  v3_decode   T=256, routed_scaling_factor 2.5, BF16 x~N(0,1), BF16 weights~N(0,0.006),
              FP8 experts, bias 0
  v3_prefill  T=16384, as v3_decode, bias~U(-0.05,0.05)
  v3_skewed   T=8192, bias = 0.5*ln(Zipf(1.2) probabilities) placed by a seeded
              permutation of the experts
  v3_top1     T=32768, top-1 routing (no renormalisation), bias 0, load-driven bias update
"""
import torch

V3 = dict(hidden=7168, inter=2048, n_experts=256, n_group=8, topk_group=4, top_k=8,
          routed_scaling_factor=2.5, has_shared=1, mode="fp8", x_std=1.0, w_std=0.006,
          seed=0)

CONFIGS = {
    "tiny_fp32": dict(T=64, hidden=256, inter=128, n_experts=16, n_group=4, topk_group=2,
                      top_k=2, routed_scaling_factor=1.0, has_shared=1, mode="fp32",
                      x_std=1.0, w_std=0.02, bias=("uniform", 0.1), seed=0,
                      update_bias=False),
    "v3_decode": dict(V3, T=256, bias=("zero",), update_bias=False),
    "v3_prefill": dict(V3, T=16384, bias=("uniform", 0.05), update_bias=False),
    "v3_skewed": dict(V3, T=8192, bias=("zipf", 1.2, 0.5), update_bias=False),
    "v3_top1": dict(V3, T=32768, top_k=1, bias=("zero",), update_bias=True),
}

# stream ids: one independent seeded generator per tensor
_X, _WG, _BIAS, _W13, _W2, _PERM = 1, 2, 3, 4, 5, 6


def config(name, **over):
    """A copy of a named workload, with fields overridden (e.g. T=512 for a cut-down case)."""
    c = dict(CONFIGS[name])
    c.update(over)
    c["name"] = name
    return c


def _gen(seed, stream, device):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed) * 1000003 + stream)
    return g


def _normal(shape, std, seed, stream, device, dtype):
    g = _gen(seed, stream, device)
    t = torch.randn(*shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t.to(dtype)


def _stacked_normal(n, shape, std, seed, stream, device, dtype):
    """n matrices of `shape`, each from its own sub-stream (bounded FP32 temporaries)."""
    out = torch.empty((n, *shape), device=device, dtype=dtype)
    for i in range(n):
        out[i] = _normal(shape, std, seed * 7919 + i, stream, device, dtype)
    return out


def bias_for(cfg):
    """Selection bias [E] float32 on the CPU."""
    E = cfg["n_experts"]
    kind = cfg["bias"][0]
    if kind == "zero":
        return torch.zeros(E, dtype=torch.float32)
    if kind == "uniform":
        a = float(cfg["bias"][1])
        g = _gen(cfg["seed"], _BIAS, "cpu")
        return (torch.rand(E, generator=g, dtype=torch.float32) * (2 * a) - a)
    if kind == "zipf":
        s, scale = float(cfg["bias"][1]), float(cfg["bias"][2])
        ranks = torch.arange(1, E + 1, dtype=torch.float64)
        p = ranks.pow(-s)
        p = p / p.sum()
        g = _gen(cfg["seed"], _PERM, "cpu")
        perm = torch.randperm(E, generator=g)
        b = torch.empty(E, dtype=torch.float64)
        b[perm] = scale * torch.log(p)
        return b.to(torch.float32)
    raise ValueError(kind)


def make_inputs(cfg, device="cpu", weights=True):
    """Draw x [T,H], Wg [E,H], bias [E] and (if weights) W13 [E+S,2I,H], W2 [E+S,H,I] on
    `device`.  The shared expert, when present, is the last slot of W13/W2.  FP32 for the
    all-FP32 workload, BF16 otherwise."""
    T, H, I, E = cfg["T"], cfg["hidden"], cfg["inter"], cfg["n_experts"]
    S = int(bool(cfg["has_shared"]))
    dt = torch.float32 if cfg["mode"] == "fp32" else torch.bfloat16
    seed = cfg["seed"]
    out = dict(
        x=_normal((T, H), cfg["x_std"], seed, _X, device, dt),
        Wg=_normal((E, H), cfg["w_std"], seed, _WG, device, dt),
        bias=bias_for(cfg).to(device),
    )
    if weights:
        out["W13"] = _stacked_normal(E + S, (2 * I, H), cfg["w_std"], seed, _W13, device, dt)
        out["W2"] = _stacked_normal(E + S, (H, I), cfg["w_std"], seed, _W2, device, dt)
    return out


def sample_tokens(T, n, seed=0):
    """A seeded sorted sample of n distinct token indices (all tokens if n >= T)."""
    if n >= T:
        return torch.arange(T, dtype=torch.int64)
    g = _gen(seed, 97, "cpu")
    return torch.sort(torch.randperm(T, generator=g)[:n]).values


def describe(cfg):
    return "%s T=%d H=%d I=%d E=%d G=%d TG=%d K=%d rsf=%g shared=%d %s" % (
        cfg.get("name", "?"), cfg["T"], cfg["hidden"], cfg["inter"], cfg["n_experts"],
        cfg["n_group"], cfg["topk_group"], cfg["top_k"], cfg["routed_scaling_factor"],
        cfg["has_shared"], cfg["mode"])

