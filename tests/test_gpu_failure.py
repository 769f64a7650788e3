"""Failure detection without a GPU fault: a bounded device wait that nothing satisfies gives up
after its clock budget, records an error word that moe_device_error returns (once), and the
context stays usable for the next launches."""
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    from fp8_gemm_sigmoid_b300 import build, moe as m
    build.build()
    assert torch.cuda.is_available()
    return m


def test_expired_wait_is_reported_and_context_survives(moe):
    assert moe.moe_device_error() == 0
    moe.moe_selftest_wait_timeout(2_000_000)  # about a millisecond of SM clock
    torch.cuda.synchronize()
    assert moe.moe_device_error() == 0x1FF
    assert moe.moe_device_error() == 0  # read once, then cleared
    # the context still runs work
    x = torch.arange(1024, device="cuda", dtype=torch.float32)
    assert float(x.sum()) == 1023 * 1024 / 2
    from fp8_gemm_sigmoid_b300 import synthetic as sy
    cfg = sy.config("tiny_fp32")
    inp = sy.make_inputs(cfg, "cuda", weights=False)
    out = moe.empty_outputs(cfg, cfg["T"])
    moe.moe_gate(cfg, inp["x"], inp["Wg"], inp["bias"], out["topk_idx"], out["topk_w"], out["counts"])
    torch.cuda.synchronize()
    assert int(out["counts"].sum()) == cfg["T"] * cfg["top_k"]
    assert moe.moe_device_error() == 0


def test_selftest_rejects_bad_budgets(moe):
    with pytest.raises(moe.MoEError):
        moe.moe_selftest_wait_timeout(0)
