"""The MOE_CHECKS debug build (libmoe_checks.so): kernels that check the indices callers pass
in, record a code in the device error word and skip the access, next to the default build on
the same inputs.  Every bad input here is one that the checks build refuses before touching
memory; the default library only gets inputs it handles (the combine skips out-of-range rows,
the gathered GEMM clamps out-of-range tokens), never unusable GEMM offsets."""
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
    build.build(checks=True)
    assert torch.cuda.is_available()
    return m


def _small_layer(moe, T=160, E=16, K=4, H=512, I=256, seed=5, mode="fp8"):
    cfg = dict(hidden=H, inter=I, n_experts=E, n_group=4, topk_group=2, top_k=K, routed_scaling_factor=2.5,
               has_shared=1, mode=mode)
    g = torch.Generator(device=DEV).manual_seed(seed)
    x = torch.randn(T, H, generator=g, device=DEV).to(torch.bfloat16)
    W13 = (torch.randn(E + 1, 2 * I, H, generator=g, device=DEV) * 0.02).to(torch.bfloat16)
    W2 = (torch.randn(E + 1, H, I, generator=g, device=DEV) * 0.02).to(torch.bfloat16)
    return cfg, x, W13, W2


def _forward(moe, cfg, x, Wg, q, T):
    out = moe.empty_outputs(cfg, T)
    bias = torch.zeros(cfg["n_experts"], dtype=torch.float32, device=DEV)
    moe.moe_forward(cfg, x.view(torch.uint16), dict(Wg=Wg.view(torch.uint16), **q), bias, 0, out["y"],
                    out["topk_idx"], out["topk_w"], out["counts"], moe.workspace(cfg, T))
    torch.cuda.synchronize()
    return {k: to_host(v) for k, v in out.items()}


@pytest.mark.parametrize("mode", ["fp8", "mxfp8"])
def test_checks_build_gives_the_default_results(moe, mode):
    """On valid inputs the checks change nothing: the whole layer forward of both libraries is
    bit-identical and records no code."""
    T = 160
    cfg, x, W13, W2 = _small_layer(moe, T=T, mode=mode)
    Wg = (torch.randn(cfg["n_experts"], cfg["hidden"], device=DEV) * 0.05).to(torch.bfloat16)
    q = moe.quantize_weights(W13, W2, pow2=mode == "mxfp8")
    ref = _forward(moe, cfg, x, Wg, q, T)
    assert moe.moe_device_error() == 0
    with moe.checks_library():
        got = _forward(moe, cfg, x, Wg, q, T)
        assert moe.moe_device_error() == 0
    for k in ref:
        assert np.array_equal(ref[k], got[k]), k


def test_combine_row_out_of_range_is_recorded_and_skipped(moe):
    T, K, H, E = 70, 4, 256, 8
    cfg = dict(hidden=H, inter=128, n_experts=E, n_group=1, topk_group=1, top_k=K, routed_scaling_factor=1.0,
               has_shared=1, mode="fp8")
    g = torch.Generator(device=DEV).manual_seed(9)
    yexp = torch.randn(T * K, H, generator=g, device=DEV).to(torch.bfloat16)
    ysh = torch.randn(T, H, generator=g, device=DEV).to(torch.bfloat16)
    w = torch.rand(T, K, generator=g, device=DEV)
    row_of = torch.randperm(T * K, generator=g, device=DEV).to(torch.int32).view(T, K)
    bad = row_of.clone()
    bad[3, 1] = T * K + 5      # past the rows
    bad[40, 2] = -9            # neither a row nor the dropped mark
    dropped = row_of.clone()
    dropped[3, 1] = -1
    dropped[40, 2] = -1
    y_ref = torch.empty(T, H, dtype=torch.bfloat16, device=DEV)
    moe.moe_combine(cfg, T, yexp, dropped, w, ysh, y_ref)
    y_def = torch.empty_like(y_ref)
    moe.moe_combine(cfg, T, yexp, bad, w, ysh, y_def)   # the default build skips them silently
    torch.cuda.synchronize()
    assert moe.moe_device_error() == 0
    with moe.checks_library():
        y_chk = torch.empty_like(y_ref)
        moe.moe_combine(cfg, T, yexp, bad, w, ysh, y_chk)
        assert moe.moe_device_error() == 0x302
        assert moe.moe_device_error() == 0          # read and cleared
        moe.moe_combine(cfg, T, yexp, dropped, w, ysh, y_chk)  # -1 is a dropped slot, not an error
        assert moe.moe_device_error() == 0
    assert torch.equal(y_def.view(torch.int16), y_ref.view(torch.int16))
    assert torch.equal(y_chk.view(torch.int16), y_ref.view(torch.int16))


@pytest.mark.parametrize("mx", [False, True])
@pytest.mark.parametrize("offs_case", ["decreasing", "past_rows", "negative"])
def test_gemm_unusable_offsets_run_no_tile(moe, mx, offs_case):
    """Group offsets that would send tiles out of the operands: the checks build records
    0x121 (FP32-scale GEMM) or 0x122 (power-of-two GEMM) and leaves the output untouched."""
    G, R, N, Kd = 3, 384, 512, 512
    g = torch.Generator(device=DEV).manual_seed(21)
    A = torch.randint(0, 120, (R, Kd), generator=g, device=DEV, dtype=torch.uint8)
    As = torch.full((Kd // 128, R), 1.0, dtype=torch.float32, device=DEV)
    W = torch.randint(0, 120, (G, N, Kd), generator=g, device=DEV, dtype=torch.uint8)
    Ws = torch.full((G, N // 128, Kd // 128), 1.0, dtype=torch.float32, device=DEV)
    offs = {"decreasing": [0, 256, 128, 384], "past_rows": [0, 128, 256, R + 256],
            "negative": [-128, 0, 128, 256]}[offs_case]
    offs = torch.tensor(offs, dtype=torch.int32, device=DEV)
    out = torch.full((R, N), 0x3f80, dtype=torch.int16, device=DEV).view(torch.bfloat16)
    with moe.checks_library():
        if mx:
            moe.moe_grouped_gemm_mxfp8(G, offs, R, N, Kd, A, As, W, Ws, moe.MOE_EPI_STORE, out, None)
        else:
            moe.moe_grouped_gemm_fp8(G, offs, R, N, Kd, A, As, W, Ws, moe.MOE_EPI_STORE, out, None, None)
        assert moe.moe_device_error() == (0x122 if mx else 0x121)
    assert bool((out.view(torch.int16) == 0x3f80).all())


@pytest.mark.parametrize("mx", [False, True])
def test_gathered_gemm_token_out_of_range(moe, mx):
    """perm_tok entries past the tokens, or negative but not -1: the checks build records 0x131
    / 0x132; both builds read such rows as zeros, the result of marking them -1."""
    T, E, K, H, I = 150, 8, 2, 512, 256
    g = torch.Generator(device=DEV).manual_seed(33 + mx)
    x = torch.randn(T, H, generator=g, device=DEV).to(torch.bfloat16)
    W13 = (torch.randn(E, 2 * I, H, generator=g, device=DEV) * 0.02).to(torch.bfloat16)
    W2 = (torch.randn(E, H, I, generator=g, device=DEV) * 0.02).to(torch.bfloat16)
    qw = moe.quantize_weights(W13, W2, pow2=mx)
    xq = torch.empty(T, H, dtype=torch.uint8, device=DEV)
    xs = torch.empty(T, H // 128, dtype=torch.float32, device=DEV)
    (moe.moe_quant_1x128_pow2 if mx else moe.moe_quant_1x128)(x.view(torch.uint16), xq, xs)
    R = T * K
    perm = torch.randint(0, T, (R,), generator=g, device=DEV, dtype=torch.int32)
    counts = np.full(E, R // E)
    counts[-1] += R - counts.sum()
    offs = torch.tensor(np.concatenate([[0], np.cumsum(counts)]), dtype=torch.int32, device=DEV)
    bad, marked = perm.clone(), perm.clone()
    for r, v in ((5, T), (77, T + 1000), (210, -4)):
        bad[r], marked[r] = v, -1

    def run(perm_tok):
        hq = torch.full((R, I), 0x55, dtype=torch.uint8, device=DEV)
        hs = torch.full((I // 128, R), 3.0, dtype=torch.float32, device=DEV)
        moe.moe_grouped_gemm_fp8_gather(E, offs, R, 2 * I, H, perm_tok, xq, xs, qw["W13"], qw["W13_s"],
                                        moe.MOE_EPI_SWIGLU_QUANT, hq, hs, mx=mx)
        torch.cuda.synchronize()
        return to_host(hq), to_host(hs)

    ref = run(marked)
    got_def = run(bad)
    assert moe.moe_device_error() == 0
    with moe.checks_library():
        got_chk = run(bad)
        assert moe.moe_device_error() == (0x132 if mx else 0x131)
    for got in (got_def, got_chk):
        assert np.array_equal(ref[0], got[0]) and np.array_equal(ref[1], got[1])
