"""GPU parity of the power-of-two (MXFP8) mode against the oracle's fp8_pow2 mode: the
quantisers bit for bit, the block-scaled grouped GEMMs within the FP8 tolerances, and the
whole layer (Insights into DeepSeek-V3 précis §3.2: scaling factors taken natively by the
tensor cores, as Blackwell's microscaling does)."""
import numpy as np
import pytest
import torch

from parity import (TOL_FP8, bf16_bits_to_f32, check_flagged_routing, check_routing, check_valid_routing,
                    rel_err, to_host)

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module")
def moe():
    from fp8_gemm_sigmoid_b300 import build, moe as m
    build.build()
    return m


@pytest.fixture(scope="module")
def sy():
    from fp8_gemm_sigmoid_b300 import synthetic
    return synthetic


def test_quant_pow2_bitexact(moe, orc):
    g = torch.Generator(device=DEV).manual_seed(31)
    rows, cols = 300, 2048
    x = torch.randn(rows, cols, generator=g, device=DEV) * 3
    x[5] = 0                                   # all-zero tiles: scale 1, codes 0
    x[6, :128] = 448.0                         # amax exactly 448 * 2^0
    x[6, 128:256] = 448.0 * 1.0078125          # one BF16 step above: the next power of two
    x[7, :128] *= 1e-35                        # tiny tiles: the 2^-127 floor
    x[8, 256:384] = 1e30                       # large constant tile
    x = x.to(torch.bfloat16).contiguous()
    q = torch.empty(rows, cols, dtype=torch.uint8, device=DEV)
    s = torch.empty(rows, cols // 128, dtype=torch.float32, device=DEV)
    moe.moe_quant_1x128_pow2(x.view(torch.uint16), q, s)
    w = (torch.randn(3, 256, 384, generator=g, device=DEV) * 0.006).to(torch.bfloat16)
    w[1, :128, :128] = 0
    w[2, 128:256, 128:256] *= 1e5
    wq = torch.empty(3, 256, 384, dtype=torch.uint8, device=DEV)
    ws = torch.empty(3, 2, 3, dtype=torch.float32, device=DEV)
    moe.moe_quant_128x128(w.contiguous().view(torch.uint16), wq, ws, pow2=True)
    torch.cuda.synchronize()
    rq, rs = orc.quant_1x128(to_host(x), pow2=True)
    assert np.array_equal(to_host(s), rs)
    assert np.array_equal(to_host(q), rq)
    rwq, rws = orc.quant_128x128(to_host(w), pow2=True)
    assert np.array_equal(to_host(ws), rws)
    assert np.array_equal(to_host(wq), rwq)
    e = np.log2(to_host(s))
    assert np.array_equal(e, np.round(e))      # every scale an exact power of two


def _groups(rng, E, total, empty=()):
    w = rng.random(E)
    for e in empty:
        w[e] = 0
    c = np.floor(w / w.sum() * total).astype(np.int64)
    c[np.argmax(w)] += total - c.sum()
    return c


# (640, 768, ...): 5 and 6 K blocks per tile, so the scale writers' four-slot stores and their
# one-slot stores alternate, and the ring position moves off and back onto a four-slot boundary
@pytest.mark.parametrize("H,I,E,R", [(384, 256, 5, 700), (7168, 2048, 4, 300), (1024, 512, 3, 257),
                                     (640, 768, 4, 400)])
def test_grouped_gemm_mxfp8_swiglu_and_down(moe, orc, H, I, E, R):
    rng = np.random.default_rng(H + R + 1)
    counts = _groups(rng, E, R, empty=(1,))
    offs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    g = torch.Generator(device=DEV).manual_seed(R + 7)
    x = torch.randn(R, H, generator=g, device=DEV).to(torch.bfloat16)
    W13 = (torch.randn(E, 2 * I, H, generator=g, device=DEV) * 0.02).to(torch.bfloat16)
    W2 = (torch.randn(E, H, I, generator=g, device=DEV) * 0.02).to(torch.bfloat16)
    aq = torch.empty(R, H, dtype=torch.uint8, device=DEV)
    as_ = torch.empty(R, H // 128, dtype=torch.float32, device=DEV)
    moe.moe_quant_1x128_pow2(x.view(torch.uint16), aq, as_)
    qw = moe.quantize_weights(W13, W2, pow2=True)
    d_offs = torch.from_numpy(offs).to(DEV)
    hq = torch.empty(R, I, dtype=torch.uint8, device=DEV)
    hs = torch.empty(I // 128, R, dtype=torch.float32, device=DEV)
    moe.moe_grouped_gemm_mxfp8(E, d_offs, R, 2 * I, H, aq, as_.t().contiguous(), qw["W13"], qw["W13_s"],
                               moe.MOE_EPI_SWIGLU_QUANT, hq, hs)
    y = torch.empty(R, H, dtype=torch.bfloat16, device=DEV)
    moe.moe_grouped_gemm_mxfp8(E, d_offs, R, H, I, hq, hs, qw["W2"], qw["W2_s"], moe.MOE_EPI_STORE, y, None)
    torch.cuda.synchronize()
    assert moe.moe_device_error() == 0
    row_e = np.repeat(np.arange(E), counts).astype(np.int32)
    rq, rs = orc.quant_1x128(to_host(x), pow2=True)
    oq = orc.quantize_weights(to_host(W13), to_host(W2), pow2=True)
    yref, aux = orc.ffn_fp8(rq, rs, row_e, *oq, want_h=True, pow2=True)
    hs_rows = to_host(hs).T
    # h's power-of-two scales: equal, except a tile whose amax sits on 448 * 2^k to within
    # the FP32 summation order may take the neighbouring power (a factor of 2)
    same_s = hs_rows == aux["hs"]
    assert same_s.mean() > 0.999
    assert np.all(np.isin(hs_rows[~same_s] / aux["hs"][~same_s], [0.5, 2.0]))
    gq, rq_h = to_host(hq), aux["hq"]
    ok_rows = np.repeat(same_s, 128, axis=1)
    diff = (gq != rq_h) & ok_rows
    assert diff.mean() < 1e-3, diff.mean()
    mag = lambda c: (c & 0x7F).astype(np.int32)  # noqa: E731
    assert np.all(np.abs(mag(gq[diff]) - mag(rq_h[diff])) <= 1)
    # the down projection of the GPU's h against the oracle's layer path
    assert rel_err(bf16_bits_to_f32(to_host(y)), bf16_bits_to_f32(yref)) <= TOL_FP8


def _layer(moe, sy, orc, cfg, n_sample):
    T = cfg["T"]
    inp = sy.make_inputs(cfg, DEV)
    q = moe.quantize_weights(inp["W13"], inp["W2"], pow2=True)
    out = moe.empty_outputs(cfg, T)
    moe.moe_forward(cfg, inp["x"].view(torch.uint16), dict(Wg=inp["Wg"].view(torch.uint16), **q),
                    inp["bias"].clone(), 0, out["y"].view(torch.uint16), out["topk_idx"], out["topk_w"],
                    out["counts"], moe.workspace(cfg, T))
    torch.cuda.synchronize()
    assert moe.moe_device_error() == 0
    sample = sy.sample_tokens(T, n_sample, seed=4).numpy()
    # the experts the sample touches, fetched from the device one set at a time
    W13 = lambda ids: to_host(inp["W13"][torch.from_numpy(np.asarray(ids)).to(DEV)])  # noqa: E731
    W2 = lambda ids: to_host(inp["W2"][torch.from_numpy(np.asarray(ids)).to(DEV)])  # noqa: E731
    ref = orc.forward(dict(cfg, mode="fp8_pow2"), to_host(inp["x"]), to_host(inp["Wg"]), to_host(inp["bias"]),
                      W13, W2, sample=sample, want_scores=True)
    gi, gw = to_host(out["topk_idx"]), to_host(out["topk_w"])
    flagged = check_routing(gi, gw, ref, cfg["routed_scaling_factor"])
    check_valid_routing(gi, cfg["n_experts"], cfg["n_group"], cfg["topk_group"])
    check_flagged_routing(gi, gw, ref, to_host(inp["bias"]), cfg["n_group"], cfg["topk_group"],
                          cfg["routed_scaling_factor"])
    same = np.all(np.sort(gi, 1) == np.sort(ref["topk_idx"], 1), axis=1)
    assert same[~flagged].all()
    keep = same[sample]
    err = rel_err(bf16_bits_to_f32(to_host(out["y"])[sample][keep]), ref["y_f32"][keep])
    assert err <= TOL_FP8, err
    return err


def test_layer_mxfp8_small(moe, sy, orc):
    """A cut-down layer (H=512, I=256, 64 experts in 2 groups of 32, top-4) on every token."""
    cfg = sy.config("v3_decode", T=300, hidden=512, inter=256, n_experts=64, n_group=2, topk_group=1,
                    top_k=4, seed=12, mode="mxfp8")
    _layer(moe, sy, orc, cfg, 300)


@pytest.mark.slow
def test_layer_mxfp8_v3_shape(moe, sy, orc):
    """The DeepSeek-V3 layer shape (H=7168, I=2048, 256 + 1 experts, top-8) at T=2048 on a
    seeded 128-token sample."""
    cfg = sy.config("v3_prefill", T=2048, seed=13, mode="mxfp8")
    _layer(moe, sy, orc, cfg, 128)
