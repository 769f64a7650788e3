"""moe_pipeline_*: the layer from and to host memory, batches overlapping.

Each batch must give exactly what moe_forward gives on the device for the same inputs (the
same kernels run; the pipeline only moves data and orders streams), including the order of
bias updates across batches and a batch smaller than the capacity."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module")
def moe():
    from fp8_gemm_sigmoid_b300 import build, moe as m
    build.build()
    assert torch.cuda.is_available()
    return m


@pytest.mark.parametrize("update_bias", [0, 1])
def test_pipeline_matches_device_forward(moe, update_bias):
    from fp8_gemm_sigmoid_b300 import synthetic as sy
    cfg = sy.config("v3_decode", T=300, hidden=512, inter=256, n_experts=16, n_group=4,
                    topk_group=2, top_k=4, seed=9)
    inp = sy.make_inputs(cfg, DEV)
    q = moe.quantize_weights(inp["W13"], inp["W2"])
    weights = dict(Wg=inp["Wg"].view(torch.uint16), **q)
    sizes = [300, 300, 177, 300]
    g = torch.Generator(device=DEV).manual_seed(3)
    xs = [torch.randn(T, 512, generator=g, device=DEV).to(torch.bfloat16) for T in sizes]

    # reference: moe_forward on the device, batch after batch
    bias_ref = inp["bias"].clone()
    ref = []
    for x in xs:
        o = moe.empty_outputs(cfg, x.shape[0])
        moe.moe_forward(cfg, x.view(torch.uint16), weights, bias_ref, update_bias, o["y"].view(torch.uint16),
                        o["topk_idx"], o["topk_w"], o["counts"], moe.workspace(cfg, x.shape[0]))
        ref.append({k: v.cpu() for k, v in o.items()})
    torch.cuda.synchronize()

    # the pipeline, from pinned host buffers
    bias = inp["bias"].clone()
    pl = moe.MoEPipeline(cfg, 300)
    outs = []
    for x in xs:
        T = x.shape[0]
        h = dict(x=x.view(torch.uint16).cpu().pin_memory(),
                 y=torch.empty(T, 512, dtype=torch.uint16).pin_memory(),
                 topk_idx=torch.empty(T, 4, dtype=torch.int32).pin_memory(),
                 topk_w=torch.empty(T, 4, dtype=torch.float32).pin_memory(),
                 counts=torch.empty(16, dtype=torch.int32).pin_memory())
        pl.submit(h["x"], weights, bias, update_bias, h["y"], h["topk_idx"], h["topk_w"], h["counts"])
        outs.append(h)
    pl.wait()
    pl.close()
    for r, h in zip(ref, outs):
        assert torch.equal(h["y"], r["y"].view(torch.uint16))
        assert torch.equal(h["topk_idx"], r["topk_idx"])
        assert torch.equal(h["topk_w"], r["topk_w"])
        assert torch.equal(h["counts"], r["counts"])
    assert torch.equal(bias.cpu(), bias_ref.cpu())
    assert moe.moe_device_error() == 0


def test_pipeline_rejects_oversized_batches(moe):
    from fp8_gemm_sigmoid_b300 import synthetic as sy
    cfg = sy.config("tiny_fp32")
    pl = moe.MoEPipeline(cfg, 8)
    x = torch.zeros(9, 256).pin_memory()
    y = torch.empty(9, 256).pin_memory()
    with pytest.raises(moe.MoEError):
        pl.submit(x, dict(Wg=torch.zeros(16, 256, device=DEV), W13=torch.zeros(1, device=DEV),
                          W2=torch.zeros(1, device=DEV)),
                  torch.zeros(16, device=DEV), 0, y, torch.empty(9, 2, dtype=torch.int32),
                  torch.empty(9, 2), torch.empty(16, dtype=torch.int32))
    pl.close()
