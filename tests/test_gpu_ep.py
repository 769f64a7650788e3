"""The expert-parallel layer (fp8_gemm_sigmoid_b300.ep.EPLayer) through libmoe on one GPU: with
a one-rank process group every exchange is the identity, so the layer must give moe_forward's
routing and output bit for bit (same rows through the same experts in the same kernels, the
shared expert on the rank's own tokens, the same combine).  More ranks need more GPUs; their
exchange logic is covered by the gloo tests."""
import os

import numpy as np
import pytest
import torch
import torch.distributed as dist

from parity import to_host

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module")
def one_rank_group():
    own = not dist.is_initialized()
    if own:
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        os.environ.setdefault("MASTER_PORT", str(29000 + os.getpid() % 1000))
        dist.init_process_group("nccl", rank=0, world_size=1)
    yield
    if own:
        dist.destroy_process_group()


@pytest.mark.parametrize("mode", ["fp8", "mxfp8"])
@pytest.mark.parametrize("E,G,TG,K,T", [(64, 2, 1, 4, 300), (16, 4, 2, 2, 129)])
def test_ep_layer_one_rank_equals_moe_forward(one_rank_group, E, G, TG, K, T, mode):
    from fp8_gemm_sigmoid_b300 import build, ep, moe, synthetic as sy
    build.build()
    torch.cuda.set_device(0)
    cfg = sy.config("v3_decode", T=T, hidden=512, inter=256, n_experts=E, n_group=G, topk_group=TG,
                    top_k=K, seed=21, mode=mode)
    inp = sy.make_inputs(cfg, DEV)
    q = moe.quantize_weights(inp["W13"], inp["W2"], pow2=mode == "mxfp8")
    x = inp["x"].view(torch.uint16)
    Wg = inp["Wg"].view(torch.uint16)
    ref = moe.empty_outputs(cfg, T)
    moe.moe_forward(cfg, x, dict(Wg=Wg, **q), inp["bias"].clone(), 0, ref["y"].view(torch.uint16),
                    ref["topk_idx"], ref["topk_w"], ref["counts"], moe.workspace(cfg, T))
    layer = ep.EPLayer(cfg, dict(Wg=Wg, **q))
    out = moe.empty_outputs(cfg, T)
    plan = layer.forward(x, inp["bias"].clone(), out["y"].view(torch.uint16), out["topk_idx"], out["topk_w"],
                         out["counts"])
    torch.cuda.synchronize()
    assert moe.moe_device_error() == 0
    assert plan["send"] == plan["recv"] == [T * K]
    for k in ("topk_idx", "topk_w", "counts"):
        assert np.array_equal(to_host(out[k]), to_host(ref[k])), k
    assert np.array_equal(to_host(out["y"]), to_host(ref["y"]))
