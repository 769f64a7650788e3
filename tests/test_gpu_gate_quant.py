"""moe_gate_quant (the gate with the 1x128 quantisation of x fused in), called through the C ABI:
its routing, weights and counts must be moe_gate's and its codes and scales moe_quant_1x128's
(moe_quant_1x128_pow2's in MXFP8 mode), bit for bit, on ragged token counts over several
tiles, with all-zero and saturating tiles.  moe_forward takes this path in both FP8 modes from
MOE_GATE_QUANT_MIN_TOKENS tokens up, so the full-size layer parity tests against the oracle
(8192 tokens and more) cover it as well, and the smaller layers cover the two kernels apart."""
import numpy as np
import pytest
import torch

from parity import to_host

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module")
def moe():
    from fp8_gemm_sigmoid_b300 import build, moe as m
    build.build()
    return m


def _inputs(T, H, E, seed):
    g = torch.Generator(device=DEV).manual_seed(seed)
    x = torch.randn(T, H, generator=g, device=DEV)
    if T > 3:
        x[1] = 0                       # every tile of the row is zero: scale 1, codes 0
        x[2, :128] *= 1e4              # large values beside small ones
        x[3, 128:256] = -3.0           # one magnitude
    if T > 4:
        # a tile of BF16 subnormals (below 2^-126), both signs: the fused kernel's packed
        # maximum must see them as the quantiser's FP32 maximum does
        x[4, 256:384] = torch.linspace(-3e-39, 5e-39, 128, device=DEV)
    x = x.to(torch.bfloat16)
    Wg = (torch.randn(E, H, generator=g, device=DEV) * 0.05).to(torch.bfloat16)
    bias = (torch.rand(E, generator=g, device=DEV) - 0.5) * 0.1
    return x, Wg, bias


@pytest.mark.parametrize("mode", ["fp8", "mxfp8"])
@pytest.mark.parametrize("T,H,E,G,TG,K", [(1, 512, 64, 2, 1, 4), (333, 512, 64, 2, 1, 4),
                                          (300, 7168, 256, 8, 4, 8), (129, 1024, 128, 4, 2, 6)])
def test_gate_quant_equals_gate_then_quant(moe, mode, T, H, E, G, TG, K):
    cfg = dict(hidden=H, inter=256, n_experts=E, n_group=G, topk_group=TG, top_k=K,
               routed_scaling_factor=2.5, has_shared=1, mode=mode)
    x, Wg, bias = _inputs(T, H, E, seed=T + E)
    xb, Wb = x.view(torch.uint16), Wg.view(torch.uint16)
    i32, f32, u8 = torch.int32, torch.float32, torch.uint8

    def outs():
        return (torch.full((T, K), -7, dtype=i32, device=DEV), torch.full((T, K), -1.0, dtype=f32, device=DEV),
                torch.full((E,), -3, dtype=i32, device=DEV), torch.full((T, H), 0x55, dtype=u8, device=DEV),
                torch.full((T, H // 128), -2.0, dtype=f32, device=DEV))

    ref = outs()
    moe.moe_gate(cfg, xb, Wb, bias, ref[0], ref[1], ref[2])
    (moe.moe_quant_1x128_pow2 if mode == "mxfp8" else moe.moe_quant_1x128)(xb, ref[3], ref[4])
    got = outs()
    moe.moe_gate_quant(cfg, xb, Wb, bias, *got)
    torch.cuda.synchronize()
    assert moe.moe_device_error() == 0
    for name, a, b in zip(("topk_idx", "topk_w", "counts", "xq", "xs"), ref, got):
        assert np.array_equal(to_host(a), to_host(b)), name
    if T > 3:
        assert not to_host(got[3])[1].any() and np.all(to_host(got[4])[1] == 1.0)


def test_gate_quant_zero_tokens_and_unsupported(moe):
    cfg = dict(hidden=512, inter=256, n_experts=64, n_group=2, topk_group=1, top_k=4,
               routed_scaling_factor=1.0, has_shared=1, mode="fp8")
    x, Wg, bias = _inputs(4, 512, 64, seed=3)
    counts = torch.full((64,), 9, dtype=torch.int32, device=DEV)
    e = torch.empty(0, dtype=torch.int32, device=DEV)
    moe.moe_gate_quant(cfg, x[:0].view(torch.uint16), Wg.view(torch.uint16), bias, e, e.float(), counts, e.byte(),
                       e.float())
    torch.cuda.synchronize()
    assert not to_host(counts).any()       # T == 0 only zeroes the counts
    bad = dict(cfg, n_group=4, topk_group=2)   # groups of 16 experts: outside the fused kernel
    with pytest.raises(moe.MoEError) as ei:
        moe.moe_gate_quant(bad, x.view(torch.uint16), Wg.view(torch.uint16), bias,
                           torch.empty(4, 4, dtype=torch.int32, device=DEV), torch.empty(4, 4, device=DEV),
                           counts, torch.empty(4, 512, dtype=torch.uint8, device=DEV),
                           torch.empty(4, 4, device=DEV))
    assert ei.value.status == moe.MOE_ERR_UNSUPPORTED


@pytest.mark.parametrize("mode", ["fp8", "mxfp8"])
def test_forward_is_the_same_across_the_fusion_threshold(moe, mode):
    """moe_forward fuses the quantisation into the gate from MOE_GATE_QUANT_MIN_TOKENS tokens
    up.  Every output row depends only on its own token, so the layer over that many tokens
    (one fused kernel) and over one token fewer (the gate and the quantiser apart) must give
    the shared tokens the same routing and the same output, bit for bit."""
    from fp8_gemm_sigmoid_b300 import synthetic as sy
    n = moe.MOE_GATE_QUANT_MIN_TOKENS
    cfg = sy.config("v3_prefill", T=n, hidden=512, inter=256, n_experts=64, n_group=2, topk_group=1,
                    top_k=4, mode=mode, seed=11)
    inp = sy.make_inputs(cfg, DEV)
    q = moe.quantize_weights(inp["W13"], inp["W2"], pow2=(mode == "mxfp8"))
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
