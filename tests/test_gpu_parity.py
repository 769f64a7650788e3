"""GPU parity: every libmoe entry point (called through the C ABI) against the CPU oracle,
on the same seeded inputs.  Tolerances are those of tests/parity.py.

Small cases span several tiles and ragged tails; the full-size workloads run in the launch
configuration the benchmark times, with the layer output checked on a seeded sample of
tokens (every output row depends only on its own token)."""
import numpy as np
import pytest
import torch

from parity import (TOL_FP32, TOL_FP8, bf16_bits_to_f32, check_flagged_routing, check_permutation,
                    check_routing, check_valid_routing, rel_err, to_host)

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="session")
def moe():
    from fp8_gemm_sigmoid_b300 import build, moe as m
    build.build()
    assert torch.cuda.is_available()
    return m


@pytest.fixture(scope="session")
def sy():
    from fp8_gemm_sigmoid_b300 import synthetic
    return synthetic


# ------------------------------------------------------------------ shared V3 weights

class V3Weights:
    """The DeepSeek-V3-shaped expert weights (seed 0), drawn once per session on the GPU and
    quantised there by moe_quant_128x128; the oracle quantises the experts it needs itself,
    lazily, from the same BF16 bits."""

    def __init__(self, moe, sy, orc):
        cfg = sy.config("v3_prefill")
        inp = sy.make_inputs(dict(cfg, T=1), DEV)
        self.W13, self.W2 = inp["W13"], inp["W2"]
        self.q = moe.quantize_weights(self.W13, self.W2)
        self.orc = orc
        self.cache = {}

    def oracle_q(self, ids):
        for e in ids:
            e = int(e)
            if e not in self.cache:
                w13 = to_host(self.W13[e:e + 1])
                w2 = to_host(self.W2[e:e + 1])
                self.cache[e] = self.orc.quantize_weights(w13, w2)
        parts = [self.cache[int(e)] for e in ids]
        return tuple(np.concatenate([p[i] for p in parts]) for i in range(4))


@pytest.fixture(scope="session")
def v3(moe, sy, orc):
    return V3Weights(moe, sy, orc)


# ------------------------------------------------------------------ quantisation

def test_quant_1x128_bitexact(moe, orc):
    g = torch.Generator(device=DEV).manual_seed(11)
    rows, cols = 333, 7168
    x = torch.randn(rows, cols, generator=g, device=DEV) * 3
    x[5] = 0                                    # all-zero tiles
    x[7, :128] = 0
    x[7, 5] = -2.5                              # single non-zero
    x[9, 128:256] *= 1e-30                      # subnormal-scale tile
    x[11, 256:384] = 1e4                        # constant tile: every code 448
    x = x.to(torch.bfloat16).contiguous()
    q = torch.empty(rows, cols, dtype=torch.uint8, device=DEV)
    s = torch.empty(rows, cols // 128, dtype=torch.float32, device=DEV)
    moe.moe_quant_1x128(x.view(torch.uint16), q, s)
    rq, rs = orc.quant_1x128(to_host(x))
    assert np.array_equal(to_host(s), rs)
    assert np.array_equal(to_host(q), rq)


def test_quant_128x128_bitexact(moe, orc):
    g = torch.Generator(device=DEV).manual_seed(12)
    w = (torch.randn(3, 384, 640, generator=g, device=DEV) * 0.006).to(torch.bfloat16)
    w[1, :128, :128] = 0
    w[2, 128:256, 256:384] *= 1000
    q = torch.empty(3, 384, 640, dtype=torch.uint8, device=DEV)
    s = torch.empty(3, 3, 5, dtype=torch.float32, device=DEV)
    moe.moe_quant_128x128(w.contiguous().view(torch.uint16), q, s)
    rq, rs = orc.quant_128x128(to_host(w))
    assert np.array_equal(to_host(s), rs)
    assert np.array_equal(to_host(q), rq)


# ------------------------------------------------------------------ gate

@pytest.mark.parametrize("name,T", [("tiny_fp32", 64), ("tiny_fp32", 1), ("v3_decode", 256),
                                    ("v3_prefill", 1000), ("v3_skewed", 777), ("v3_top1", 515)])
def test_gate_routing(moe, sy, orc, name, T):
    cfg = sy.config(name, T=T)
    inp = sy.make_inputs(cfg, DEV, weights=False)
    out = moe.empty_outputs(cfg, T)
    x = inp["x"].view(torch.uint16) if cfg["mode"] == "fp8" else inp["x"]
    Wg = inp["Wg"].view(torch.uint16) if cfg["mode"] == "fp8" else inp["Wg"]
    moe.moe_gate(cfg, x, Wg, inp["bias"], out["topk_idx"], out["topk_w"], out["counts"])
    torch.cuda.synchronize()
    ref = orc.gate(to_host(inp["x"]), to_host(inp["Wg"]), to_host(inp["bias"]), cfg["n_group"],
                   cfg["topk_group"], cfg["top_k"], cfg["routed_scaling_factor"], want_scores=True)
    gi, gw = to_host(out["topk_idx"]), to_host(out["topk_w"])
    flagged = check_routing(gi, gw, ref, cfg["routed_scaling_factor"])
    check_valid_routing(gi, cfg["n_experts"], cfg["n_group"], cfg["topk_group"])
    check_flagged_routing(gi, gw, ref, to_host(inp["bias"]), cfg["n_group"], cfg["topk_group"],
                          cfg["routed_scaling_factor"])
    counts = to_host(out["counts"])
    assert np.array_equal(counts, np.bincount(gi.ravel(), minlength=cfg["n_experts"]))
    if not flagged.any():
        assert np.array_equal(counts, np.bincount(ref["topk_idx"].ravel(), minlength=cfg["n_experts"]))


def test_gate_ties_and_forced_experts(moe, orc):
    """All logits equal: ties go to the lower index; then a large bias forces one group and
    experts (selection follows the bias, weights stay the un-biased scores)."""
    cfg = dict(hidden=256, inter=128, n_experts=16, n_group=4, topk_group=2, top_k=3,
               routed_scaling_factor=1.0, has_shared=0, mode="fp32")
    T = 40
    x = torch.ones(T, 256, device=DEV)
    Wg = torch.zeros(16, 256, device=DEV)
    bias = torch.zeros(16, device=DEV)
    out = moe.empty_outputs(cfg, T)
    moe.moe_gate(cfg, x, Wg, bias, out["topk_idx"], out["topk_w"], out["counts"])
    torch.cuda.synchronize()
    assert to_host(out["topk_idx"]).tolist() == [[0, 1, 2]] * T
    assert np.allclose(to_host(out["topk_w"]), 1 / 3, rtol=1e-6)
    bias[[13, 14, 9]] = torch.tensor([3.0, 2.0, 1.0], device=DEV)
    moe.moe_gate(cfg, x, Wg, bias, out["topk_idx"], out["topk_w"], out["counts"])
    torch.cuda.synchronize()
    assert to_host(out["topk_idx"]).tolist() == [[13, 14, 9]] * T
    assert np.allclose(to_host(out["topk_w"]), 1 / 3, rtol=1e-6)
    assert to_host(out["counts"]).tolist() == [0] * 9 + [T, 0, 0, 0, T, T, 0]


# ------------------------------------------------------------------ permutation

# (500, 96, 6, 1): an expert count that does not divide the scan's 1024 threads;
# (300, 1024, 32, 1): top_k * experts too large for the match kernel's shared-memory counts,
# so the positions come from the one-thread-per-expert fallback.
@pytest.mark.parametrize("T,E,K,S", [(1, 16, 2, 1), (300, 256, 8, 1), (4097, 256, 8, 0),
                                     (129, 16, 2, 1), (1000, 256, 1, 1), (500, 96, 6, 1),
                                     (300, 1024, 32, 1)])
def test_permute_bitexact(moe, orc, T, E, K, S):
    rng = np.random.default_rng(T + E + K)
    # skewed synthetic routing: some experts empty, one hot expert
    p = rng.dirichlet(np.full(E, 0.3))
    p[3] += 2.0
    p /= p.sum()
    idx = np.stack([rng.choice(E, K, replace=False, p=p) for _ in range(T)]).astype(np.int32)
    G, TG = {256: (8, 4), 1024: (32, 32)}.get(E, (4, 2))
    cfg = dict(hidden=256, inter=128, n_experts=E, n_group=G, topk_group=TG, top_k=K,
               routed_scaling_factor=1.0, has_shared=S, mode="fp8")
    H = cfg["hidden"]
    g = torch.Generator(device=DEV).manual_seed(T)
    xq = torch.randint(0, 255, (T, H), generator=g, device=DEV, dtype=torch.uint8)
    xs = torch.rand(T, H // 128, generator=g, device=DEV)
    R = T * K + T * S
    d_idx = torch.from_numpy(idx).to(DEV)
    counts = torch.from_numpy(np.bincount(idx.ravel(), minlength=E).astype(np.int32)).to(DEV)
    offs = torch.empty(E + 1 + S, dtype=torch.int32, device=DEV)
    perm_tok = torch.empty(R, dtype=torch.int32, device=DEV)
    row_of = torch.empty(T, K, dtype=torch.int32, device=DEV)
    aq = torch.empty(R, H, dtype=torch.uint8, device=DEV)
    as_ = torch.empty(H // 128, R, dtype=torch.float32, device=DEV)  # K-block-major
    ws = moe.workspace(cfg, T)
    moe.moe_permute(cfg, T, d_idx, counts, xq, xs, offs, perm_tok, row_of, aq, as_, ws)
    torch.cuda.synchronize()
    ref = check_permutation(dict(offs=to_host(offs), perm_tok=to_host(perm_tok), row_of=to_host(row_of)),
                            idx, orc, E, S)
    assert np.array_equal(to_host(aq), to_host(xq)[ref["perm_tok"]])
    assert np.array_equal(to_host(as_), to_host(xs)[ref["perm_tok"]].T)


@pytest.mark.parametrize("mode", ["fp8", "fp32"])
def test_permute_and_combine_with_dropped_ids(moe, orc, mode):
    """Expert ids outside [0, E) (never written by moe_gate, but a caller may chain the public
    calls on its own routing): the permutation drops those slots (row_of -1), zeroes the rows
    they leave unclaimed, and the combine skips them, all as the oracle's contract says."""
    T, E, K, S, H = 200, 16, 4, 1, 256
    rng = np.random.default_rng(77)
    idx = np.stack([rng.choice(E, K, replace=False) for _ in range(T)]).astype(np.int32)
    idx[3, 2] = -1
    idx[17, 0] = E
    idx[150] = [-1, 1 << 30, -7, 99]
    cfg = dict(hidden=H, inter=128, n_experts=E, n_group=4, topk_group=2, top_k=K,
               routed_scaling_factor=1.0, has_shared=S, mode=mode)
    g = torch.Generator(device=DEV).manual_seed(8)
    R = T * K + T * S
    if mode == "fp8":
        xq = torch.randint(0, 255, (T, H), generator=g, device=DEV, dtype=torch.uint8)
        xs = torch.rand(T, H // 128, generator=g, device=DEV)
        aq = torch.full((R, H), 0x7F, dtype=torch.uint8, device=DEV)       # stale NaN codes
        as_ = torch.full((H // 128, R), 7.0, dtype=torch.float32, device=DEV)
    else:
        xq = torch.randn(T, H, generator=g, device=DEV)
        xs = as_ = None
        aq = torch.full((R, H), float("nan"), dtype=torch.float32, device=DEV)
    offs = torch.empty(E + 1 + S, dtype=torch.int32, device=DEV)
    perm_tok = torch.empty(R, dtype=torch.int32, device=DEV)
    row_of = torch.empty(T, K, dtype=torch.int32, device=DEV)
    moe.moe_permute(cfg, T, torch.from_numpy(idx).to(DEV), None, xq, xs, offs, perm_tok, row_of, aq, as_,
                    moe.workspace(cfg, T))
    torch.cuda.synchronize()
    ref = check_permutation(dict(offs=to_host(offs), perm_tok=to_host(perm_tok), row_of=to_host(row_of)),
                            idx, orc, E, S)
    claimed = ref["perm_tok"] >= 0
    V = int((ref["row_of"] >= 0).sum())
    assert not claimed[V:T * K].any() and claimed[:V].all()
    assert np.array_equal(to_host(aq)[claimed], to_host(xq)[ref["perm_tok"][claimed]])
    assert not to_host(aq)[~claimed].any()      # unclaimed rows: all-zero payload
    if mode == "fp8":
        assert np.array_equal(to_host(as_)[:, claimed], to_host(xs)[ref["perm_tok"][claimed]].T)
        assert not to_host(as_)[:, ~claimed].any()
    # combine on that routing: the dropped slots add nothing
    dt = torch.bfloat16 if mode == "fp8" else torch.float32
    yexp = torch.randn(T * K, H, generator=g, device=DEV).to(dt)
    ysh = torch.randn(T, H, generator=g, device=DEV).to(dt)
    w = rng.random((T, K)).astype(np.float32)
    y = torch.empty(T, H, dtype=dt, device=DEV)
    moe.moe_combine(cfg, T, yexp, row_of, torch.from_numpy(w).to(DEV), ysh, y)
    torch.cuda.synchronize()
    drop = ref["row_of"] < 0
    yk = to_host(yexp)[np.where(drop, 0, ref["row_of"])]
    yk[drop] = 0                     # a zero term with weight 0 adds exactly nothing (y != -0)
    acc = orc.combine(yk, np.where(drop, 0, w).astype(np.float32), to_host(ysh))
    want = orc.round_bf16(acc) if mode == "fp8" else acc
    assert np.array_equal(to_host(y), want)


# ------------------------------------------------------------------ grouped expert GEMMs

def _random_groups(rng, E, total, empty=()):
    w = rng.random(E)
    for e in empty:
        w[e] = 0
    c = np.floor(w / w.sum() * total).astype(np.int64)
    c[np.argmax(w)] += total - c.sum()
    return c


# (1024, 256, 24, 400): fewer than 64 rows per group on average, the 4-stage ring with every
# output row stored directly (some groups still hold more than 32 rows)
@pytest.mark.parametrize("H,I,E,R", [(384, 256, 5, 700), (640, 384, 3, 400), (7168, 2048, 4, 300),
                                     (1024, 256, 24, 400)])
def test_grouped_gemm_fp8_swiglu_and_down(moe, orc, H, I, E, R):
    rng = np.random.default_rng(H + R)
    counts = _random_groups(rng, E, R, empty=(1,))
    offs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    g = torch.Generator(device=DEV).manual_seed(R)
    x = torch.randn(R, H, generator=g, device=DEV).to(torch.bfloat16)
    W13 = (torch.randn(E, 2 * I, H, generator=g, device=DEV) * 0.02).to(torch.bfloat16)
    W2 = (torch.randn(E, H, I, generator=g, device=DEV) * 0.02).to(torch.bfloat16)
    aq = torch.empty(R, H, dtype=torch.uint8, device=DEV)
    as_ = torch.empty(R, H // 128, dtype=torch.float32, device=DEV)
    moe.moe_quant_1x128(x.view(torch.uint16), aq, as_)
    as_k = as_.t().contiguous()  # the GEMM reads K-block-major scales
    qw = moe.quantize_weights(W13, W2)
    d_offs = torch.from_numpy(offs).to(DEV)
    hq = torch.empty(R, I, dtype=torch.uint8, device=DEV)
    hs = torch.empty(I // 128, R, dtype=torch.float32, device=DEV)  # written K-block-major
    ws = torch.empty(64 << 20 if R * 2 * I * 4 < (60 << 20) else R * 2 * I * 4 + (4 << 20),
                     dtype=torch.uint8, device=DEV)
    moe.moe_grouped_gemm_fp8(E, d_offs, R, 2 * I, H, aq, as_k, qw["W13"], qw["W13_s"],
                             moe.MOE_EPI_SWIGLU_QUANT, hq, hs, ws)
    y = torch.empty(R, H, dtype=torch.bfloat16, device=DEV)
    moe.moe_grouped_gemm_fp8(E, d_offs, R, H, I, hq, hs, qw["W2"], qw["W2_s"], moe.MOE_EPI_STORE,
                             y, None, ws)
    torch.cuda.synchronize()
    # oracle: the same rows through the same experts
    row_e = np.repeat(np.arange(E), counts).astype(np.int32)
    rq, rs = orc.quant_1x128(to_host(x))
    oq = orc.quantize_weights(to_host(W13), to_host(W2))
    yref, aux = orc.ffn_fp8(rq, rs, row_e, *oq, want_h=True)
    table = orc.e4m3_table()
    hs_rows = to_host(hs).T
    h_gpu = table[to_host(hq)] * np.repeat(hs_rows, 128, axis=1)
    h_ref = aux["h"].astype(np.float64)
    # GEMM1 + SwiGLU + 1x128 quantisation: within one code step of the oracle's FP32 h
    assert np.allclose(hs_rows, aux["hs"], rtol=1e-5, atol=0)
    step = np.repeat(aux["hs"], 128, axis=1) * 32.0  # largest E4M3 step (256..448) in code units
    assert np.all(np.abs(h_gpu - h_ref) <= step * 0.5 + 1e-30)
    # the codes themselves agree except where h sits on a rounding boundary (FP32 sums in
    # another order): at most one code step apart, and rarely
    gq, rq_h = to_host(hq), aux["hq"]
    diff = gq != rq_h
    assert diff.mean() < 1e-3, diff.mean()
    mag = lambda c: (c & 0x7F).astype(np.int32)  # noqa: E731  (codes ordered by magnitude)
    assert np.all(np.abs(mag(gq[diff]) - mag(rq_h[diff])) <= 1)
    # GEMM2 on the GPU's own h, against the oracle's layer path
    assert rel_err(bf16_bits_to_f32(to_host(y)), bf16_bits_to_f32(yref)) <= TOL_FP8


def test_grouped_gemm_f32(moe, orc):
    rng = np.random.default_rng(3)
    H, I, E, R = 256, 128, 6, 333
    counts = _random_groups(rng, E, R, empty=(0, 4))
    offs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    g = torch.Generator(device=DEV).manual_seed(5)
    x = torch.randn(R, H, generator=g, device=DEV)
    W13 = torch.randn(E, 2 * I, H, generator=g, device=DEV) * 0.05
    W2 = torch.randn(E, H, I, generator=g, device=DEV) * 0.05
    d_offs = torch.from_numpy(offs).to(DEV)
    h = torch.empty(R, I, device=DEV)
    y = torch.empty(R, H, device=DEV)
    ws = torch.empty(R * 2 * I * 4 + (1 << 20), dtype=torch.uint8, device=DEV)
    moe.moe_grouped_gemm_f32(E, d_offs, R, 2 * I, H, x, W13, moe.MOE_EPI_SWIGLU_QUANT, h, ws)
    moe.moe_grouped_gemm_f32(E, d_offs, R, H, I, h, W2, moe.MOE_EPI_STORE, y, ws)
    torch.cuda.synchronize()
    row_e = np.repeat(np.arange(E), counts).astype(np.int32)
    yref, href = orc.ffn_f32(to_host(x), row_e, to_host(W13), to_host(W2), want_h=True)
    assert rel_err(to_host(h), href) <= TOL_FP32
    assert rel_err(to_host(y), yref) <= TOL_FP32


# ------------------------------------------------------------------ combine, bias update

# BF16 rows: K = 4..8 take the kernel that issues every slot's load first, other K the general one
@pytest.mark.parametrize("mode,T,K,S", [("fp8", 300, 8, 1), ("fp8", 64, 1, 0), ("fp32", 64, 2, 1),
                                        ("fp8", 100, 6, 0), ("fp8", 70, 3, 1)])
def test_combine_bitexact(moe, orc, mode, T, K, S):
    H = 7168 if mode == "fp8" else 256
    cfg = dict(hidden=H, inter=128, n_experts=16, n_group=4, topk_group=2, top_k=K,
               routed_scaling_factor=1.0, has_shared=S, mode=mode)
    R = T * K + T * S
    g = torch.Generator(device=DEV).manual_seed(T * K)
    yexp = torch.randn(R, H, generator=g, device=DEV)
    if mode == "fp8":
        yexp = yexp.to(torch.bfloat16)
    rng = np.random.default_rng(T)
    row_of = rng.permutation(T * K).reshape(T, K).astype(np.int32)
    w = rng.random((T, K)).astype(np.float32)
    y = torch.empty(T, H, dtype=yexp.dtype, device=DEV)
    yexp = yexp.contiguous()
    ysh_d = yexp[T * K:] if S else None  # the shared expert's rows, passed as their own operand
    moe.moe_combine(cfg, T, yexp, torch.from_numpy(row_of).to(DEV), torch.from_numpy(w).to(DEV), ysh_d, y)
    torch.cuda.synchronize()
    yh = to_host(yexp)
    yk = yh[row_of]                                   # [T, K, H]
    ysh = yh[T * K:] if S else None
    acc = orc.combine(yk, w, ysh)
    ref = orc.round_bf16(acc) if mode == "fp8" else acc
    assert np.array_equal(to_host(y), ref)


def test_bias_update_bitexact(moe, orc):
    cfg = dict(hidden=256, inter=128, n_experts=256, n_group=8, topk_group=4, top_k=1,
               routed_scaling_factor=2.5, has_shared=1, mode="fp8")
    rng = np.random.default_rng(9)
    T = 32768
    counts = rng.multinomial(T, np.full(256, 1 / 256)).astype(np.int32)
    counts[:4] = T // 256   # exactly at the mean
    bias = rng.uniform(-0.1, 0.1, 256).astype(np.float32)
    d_b = torch.from_numpy(bias).to(DEV)
    moe.moe_bias_update(cfg, T, torch.from_numpy(counts).to(DEV), d_b)
    torch.cuda.synchronize()
    assert np.array_equal(to_host(d_b), orc.bias_update(counts, bias, T, 1))


# ------------------------------------------------------------------ the whole layer

def _run_forward(moe, sy, cfg, v3=None):
    T = cfg["T"]
    inp = sy.make_inputs(cfg, DEV, weights=(v3 is None))
    if cfg["mode"] == "fp8":
        if v3 is None:
            q = moe.quantize_weights(inp["W13"], inp["W2"])
        else:
            q = v3.q
        weights = dict(Wg=inp["Wg"].view(torch.uint16), **q)
        x = inp["x"].view(torch.uint16)
    else:
        weights = dict(Wg=inp["Wg"], W13=inp["W13"], W2=inp["W2"])
        x = inp["x"]
    out = moe.empty_outputs(cfg, T)
    bias = inp["bias"].clone()
    ws = moe.workspace(cfg, T)
    y = out["y"].view(torch.uint16) if cfg["mode"] == "fp8" else out["y"]
    moe.moe_forward(cfg, x, weights, bias, cfg["update_bias"], y, out["topk_idx"], out["topk_w"],
                    out["counts"], ws)
    torch.cuda.synchronize()
    assert moe.moe_device_error() == 0
    return inp, out, bias


def _check_layer(moe, sy, orc, cfg, n_sample, v3=None):
    inp, out, new_bias = _run_forward(moe, sy, cfg, v3)
    T = cfg["T"]
    sample = sy.sample_tokens(T, n_sample, seed=1).numpy()
    if v3 is None:
        W13, W2, qfn = to_host(inp["W13"]), to_host(inp["W2"]), None
    else:
        W13 = W2 = None
        qfn = v3.oracle_q
    ref = orc.forward(cfg, to_host(inp["x"]), to_host(inp["Wg"]), to_host(inp["bias"]), W13, W2,
                      sample=sample, qweights=qfn, want_scores=True)
    gi, gw = to_host(out["topk_idx"]), to_host(out["topk_w"])
    flagged = check_routing(gi, gw, ref, cfg["routed_scaling_factor"])
    check_valid_routing(gi, cfg["n_experts"], cfg["n_group"], cfg["topk_group"])
    check_flagged_routing(gi, gw, ref, to_host(inp["bias"]), cfg["n_group"], cfg["topk_group"],
                          cfg["routed_scaling_factor"])
    counts = to_host(out["counts"])
    assert np.array_equal(counts, np.bincount(gi.ravel(), minlength=cfg["n_experts"]))
    same = np.all(np.sort(gi, 1) == np.sort(ref["topk_idx"], 1), axis=1)
    assert same[~flagged].all()  # (check_routing) only flagged tokens may choose otherwise
    if same.all():
        assert np.array_equal(counts, ref["counts"])
    if cfg["update_bias"]:
        old_b = to_host(inp["bias"])
        want = orc.bias_update(ref["counts"], old_b, T, cfg["top_k"])
        got = to_host(new_bias)
        if same.all():
            assert np.array_equal(got, want)
        else:
            # a flagged token chose another valid expert: the experts whose load differs from
            # the oracle's may move another way (up, down or not at all, by one step); every
            # other expert moves exactly as the oracle's update says
            moved = counts != ref["counts"]
            assert np.array_equal(got[~moved], want[~moved])
            step = np.float32(1e-3)
            for o, g in zip(old_b[moved], got[moved]):
                assert g in (o + step, o, o - step)
    # the layer output on every sampled token whose routing is the oracle's: all the tokens
    # the oracle does not flag, and the flagged ones that chose the same experts.  The BF16
    # output is compared with the oracle's FP32 sums before their own rounding to BF16 (the
    # exact value the output format rounds), so that a single rounding, the GPU's, counts.
    keep = same[sample]
    y = to_host(out["y"])[sample][keep]
    if cfg["mode"] == "fp8":
        err = rel_err(bf16_bits_to_f32(y), ref["y_f32"][keep])
        assert err <= TOL_FP8, err
    else:
        err = rel_err(y, ref["y"][keep])
        assert err <= TOL_FP32, err
    return dict(flagged=int(flagged.sum()), err=err, counts=counts, compared=int(keep.sum()))


def test_layer_tiny_fp32(moe, sy, orc):
    cfg = sy.config("tiny_fp32")
    r = _check_layer(moe, sy, orc, cfg, n_sample=64)
    assert r["counts"].sum() == 64 * 2


@pytest.mark.parametrize("T", [1, 37, 300])
def test_layer_tiny_fp32_ragged(moe, sy, orc, T):
    _check_layer(moe, sy, orc, sy.config("tiny_fp32", T=T, seed=T), n_sample=T)


def test_layer_fp8_small_shape(moe, sy, orc):
    """A cut-down FP8 layer (H=512, I=256, 16 experts) checked on every token."""
    cfg = sy.config("v3_decode", T=300, hidden=512, inter=256, n_experts=16, n_group=4,
                    topk_group=2, top_k=4, seed=3)
    _check_layer(moe, sy, orc, cfg, n_sample=300)


def test_layer_fp8_empty_and_full_experts(moe, sy, orc):
    """A large bias forces every token onto the same 4 experts: the other groups stay empty
    and one group holds every token (several tiles and a ragged tail)."""
    cfg = sy.config("v3_decode", T=333, hidden=512, inter=256, n_experts=16, n_group=4,
                    topk_group=2, top_k=4, seed=4)
    inp, out, _ = _run_forward(moe, sy, dict(cfg, bias=("zero",)))
    # rerun with a forcing bias through the oracle and the GPU
    E = 16
    bias = np.zeros(E, np.float32)
    bias[[5, 6, 9, 10]] = 5.0
    x, Wg = inp["x"], inp["Wg"]
    q = moe.quantize_weights(inp["W13"], inp["W2"])
    o = moe.empty_outputs(cfg, 333)
    ws = moe.workspace(cfg, 333)
    moe.moe_forward(cfg, x.view(torch.uint16), dict(Wg=Wg.view(torch.uint16), **q),
                    torch.from_numpy(bias).to(DEV), 0, o["y"].view(torch.uint16), o["topk_idx"],
                    o["topk_w"], o["counts"], ws)
    torch.cuda.synchronize()
    ref = orc.forward(cfg, to_host(x), to_host(Wg), bias, to_host(inp["W13"]), to_host(inp["W2"]))
    counts = to_host(o["counts"])
    assert counts.tolist() == ref["counts"].tolist()
    assert sorted(np.nonzero(counts)[0].tolist()) == [5, 6, 9, 10]
    assert rel_err(bf16_bits_to_f32(to_host(o["y"])), ref["y_f32"]) <= TOL_FP8


def test_layer_fp8_zero_tokens(moe, sy, orc):
    cfg = sy.config("v3_decode", T=64, hidden=512, inter=256, n_experts=16, n_group=4,
                    topk_group=2, top_k=4, seed=5)
    inp = sy.make_inputs(cfg, DEV)
    inp["x"][3] = 0          # amax == 0 tiles for one token
    inp["x"][4, :128] = 0
    inp["x"][4, 7] = 1e4     # one huge value: its code is 448, the rest of the tile ~0
    q = moe.quantize_weights(inp["W13"], inp["W2"])
    o = moe.empty_outputs(cfg, 64)
    moe.moe_forward(cfg, inp["x"].view(torch.uint16), dict(Wg=inp["Wg"].view(torch.uint16), **q),
                    inp["bias"].clone(), 0, o["y"].view(torch.uint16), o["topk_idx"], o["topk_w"],
                    o["counts"], moe.workspace(cfg, 64))
    torch.cuda.synchronize()
    ref = orc.forward(cfg, to_host(inp["x"]), to_host(inp["Wg"]), to_host(inp["bias"]),
                      to_host(inp["W13"]), to_host(inp["W2"]))
    check_routing(to_host(o["topk_idx"]), to_host(o["topk_w"]), ref, cfg["routed_scaling_factor"])
    assert rel_err(bf16_bits_to_f32(to_host(o["y"])), ref["y_f32"]) <= TOL_FP8
    # T = 0: nothing but a zeroed histogram
    e = moe.empty_outputs(cfg, 0)
    e["counts"].fill_(7)
    moe.moe_forward(cfg, inp["x"][:0].view(torch.uint16), dict(Wg=inp["Wg"].view(torch.uint16), **q),
                    inp["bias"].clone(), 0, e["y"].view(torch.uint16), e["topk_idx"], e["topk_w"],
                    e["counts"], moe.workspace(cfg, 1))
    torch.cuda.synchronize()
    assert not to_host(e["counts"]).any()


@pytest.mark.slow
@pytest.mark.parametrize("name,n_sample", [("v3_decode", 256), ("v3_prefill", 512), ("v3_skewed", 512),
                                           ("v3_top1", 512)])
def test_layer_v3_full_size(moe, sy, orc, v3, name, n_sample):
    """The four DeepSeek-V3-shaped workloads at full size through moe_forward (the call the
    benchmark times): routing of every token, and the layer output on a seeded sample of 512
    tokens (all 256 for the decode batch)."""
    cfg = sy.config(name)
    r = _check_layer(moe, sy, orc, cfg, n_sample=n_sample, v3=v3)
    print("%s: flagged=%d compared=%d rel_err=%.3g nonempty_experts=%d max_count=%d" % (
        name, r["flagged"], r["compared"], r["err"], int((r["counts"] > 0).sum()), int(r["counts"].max())))


@pytest.mark.parametrize("mx", [False, True])
def test_gathered_gemm_equals_the_permuted_copy(moe, orc, mx):
    """[P1] §2.3's permuted copy of the tokens, fused away: the gate/up GEMM reading its rows
    from the quantised tokens through perm_tok gives the bytes the same GEMM gives on the
    permutation's copy, including rows no (token, slot) claims (expert ids out of range)."""
    T, E, K, H, I = 333, 16, 4, 512, 256
    rng = np.random.default_rng(55 + mx)
    idx = np.stack([rng.choice(E, K, replace=False) for _ in range(T)]).astype(np.int32)
    idx[7, 1] = -1
    idx[200, 3] = E + 3
    cfg = dict(hidden=H, inter=I, n_experts=E, n_group=4, topk_group=2, top_k=K, routed_scaling_factor=1.0,
               has_shared=1, mode="mxfp8" if mx else "fp8")
    g = torch.Generator(device=DEV).manual_seed(3 + mx)
    x = torch.randn(T, H, generator=g, device=DEV).to(torch.bfloat16)
    W13 = (torch.randn(E + 1, 2 * I, H, generator=g, device=DEV) * 0.02).to(torch.bfloat16)
    W2 = (torch.randn(E + 1, H, I, generator=g, device=DEV) * 0.02).to(torch.bfloat16)
    qw = moe.quantize_weights(W13, W2, pow2=mx)
    xq = torch.empty(T, H, dtype=torch.uint8, device=DEV)
    xs = torch.empty(T, H // 128, dtype=torch.float32, device=DEV)
    (moe.moe_quant_1x128_pow2 if mx else moe.moe_quant_1x128)(x.view(torch.uint16), xq, xs)
    R = T * K + T
    offs = torch.empty(E + 2, dtype=torch.int32, device=DEV)
    perm_tok = torch.empty(R, dtype=torch.int32, device=DEV)
    row_of = torch.empty(T, K, dtype=torch.int32, device=DEV)
    aq = torch.empty(R, H, dtype=torch.uint8, device=DEV)
    as_ = torch.empty(H // 128, R, dtype=torch.float32, device=DEV)
    moe.moe_permute(cfg, T, torch.from_numpy(idx).to(DEV), None, xq, xs, offs, perm_tok, row_of, aq, as_,
                    moe.workspace(cfg, T))
    outs = []
    for gathered in (False, True):
        hq = torch.full((R, I), 0x55, dtype=torch.uint8, device=DEV)
        hs = torch.full((I // 128, R), 3.0, dtype=torch.float32, device=DEV)
        if gathered:
            moe.moe_grouped_gemm_fp8_gather(E + 1, offs, R, 2 * I, H, perm_tok, xq, xs, qw["W13"], qw["W13_s"],
                                            moe.MOE_EPI_SWIGLU_QUANT, hq, hs, mx=mx)
        elif mx:
            moe.moe_grouped_gemm_mxfp8(E + 1, offs, R, 2 * I, H, aq, as_, qw["W13"], qw["W13_s"],
                                       moe.MOE_EPI_SWIGLU_QUANT, hq, hs)
        else:
            moe.moe_grouped_gemm_fp8(E + 1, offs, R, 2 * I, H, aq, as_, qw["W13"], qw["W13_s"],
                                     moe.MOE_EPI_SWIGLU_QUANT, hq, hs, None)
        torch.cuda.synchronize()
        outs.append((to_host(hq), to_host(hs)))
    assert moe.moe_device_error() == 0
    assert np.array_equal(outs[0][0], outs[1][0])
    assert np.array_equal(outs[0][1], outs[1][1])
    unclaimed = to_host(perm_tok) < 0
    assert unclaimed.sum() == 2 and not outs[1][0][unclaimed].any()


def test_forward_is_the_same_across_the_ring_depth_switch(moe, sy):
    """The FP32-scale grouped GEMMs take a 4-stage operand ring (and store every down-GEMM row
    directly) when the groups hold fewer than 64 rows on average, R < 64 * (E + 1).  Each
    output element's sums run in the same order either way, and each output row depends only
    on its own token, so the layer just above and just below the switch gives the shared tokens
    the same routing and output, bit for bit."""
    E, K = 64, 4
    n = 64 * (E + 1) // (K + 1)          # T(K + 1) >= 64 (E + 1): the 3-stage ring
    assert n * (K + 1) >= 64 * (E + 1) > (n - 1) * (K + 1)
    cfg = sy.config("v3_prefill", T=n, hidden=512, inter=256, n_experts=E, n_group=2, topk_group=1,
                    top_k=K, seed=12)
    inp = sy.make_inputs(cfg, DEV)
    q = moe.quantize_weights(inp["W13"], inp["W2"])
    w = dict(Wg=inp["Wg"].view(torch.uint16), **q)
    res = []
    for T in (n, n - 1):
        out = moe.empty_outputs(cfg, T)
        ws = moe.workspace(cfg, T)
        moe.moe_forward(cfg, inp["x"][:T].view(torch.uint16), w, inp["bias"].clone(), 0,
                        out["y"].view(torch.uint16), out["topk_idx"], out["topk_w"], out["counts"], ws)
        torch.cuda.synchronize()
        res.append({k: to_host(v)[: n - 1] for k, v in out.items() if k != "counts"})
    assert moe.moe_device_error() == 0
    for k in res[0]:
        assert np.array_equal(res[0][k], res[1][k]), k


@pytest.mark.slow
@pytest.mark.parametrize("name", ["v3_decode", "v3_skewed", "v3_top1"])
def test_forward_is_deterministic(moe, sy, v3, name):
    """The layer at full size, run twice on the same inputs, gives the same bytes: routing,
    weights, histogram, updated bias and output.  No atomic operation decides a value (the
    histogram's atomic adds commute), and every sum has a fixed order.  The skewed workload
    sends every token to one expert (the most contended histogram bin and the largest group);
    the top-1 workload updates the bias."""
    cfg = sy.config(name)
    runs = [_run_forward(moe, sy, cfg, v3) for _ in range(2)]
    for k in ("y", "topk_idx", "topk_w", "counts"):
        assert np.array_equal(to_host(runs[0][1][k]), to_host(runs[1][1][k])), k
    assert np.array_equal(to_host(runs[0][2]), to_host(runs[1][2]))  # the updated bias
