"""GPU parity of the LogFMT-nBit codec (moe_logfmt_encode / moe_logfmt_decode, called through
the C ABI) against the oracle (Insights into DeepSeek-V3 précis §3.2).

The code of a value is an integer decided in floating point, so both sides decide it with
their own logarithms: the codes must be equal wherever the oracle's decision margin (the
distance to the linear midpoint between two grid values, as a fraction of their gap) exceeds
MARGIN, and within one step elsewhere; the tile metadata (FP32 min and Step) must agree to a
few units in the last place."""
import numpy as np
import pytest
import torch

from parity import to_host

pytestmark = pytest.mark.gpu

DEV = "cuda"
MARGIN = 1e-3


@pytest.fixture(scope="module")
def moe():
    from fp8_gemm_sigmoid_b300 import build, moe as m
    build.build()
    return m


def _payload(rows, cols, seed):
    """Gaussian rows with per-row scales and, in the first tiles of rows 1-5, the special
    cases of the code (cols >= 256)."""
    g = torch.Generator(device=DEV).manual_seed(seed)
    x = torch.randn(rows, cols, generator=g, device=DEV)
    x = x * torch.exp(torch.randn(rows, 1, generator=g, device=DEV) * 2)   # per-row scale
    x[1, :128] = 0                                      # all-zero tile
    x[2, 128:256] = 0.75                                # one magnitude
    x[2, 130] = -0.75
    x[3, :128] *= 1e-20                                 # a tiny value beside the tile's max...
    x[3, 0] = 3.0                                       # ...so min is held at max - ln 2^32
    x[4, 128:256] = -0.0
    x[5, :128] = torch.randn(128, generator=g, device=DEV) * 1e-30  # values near the BF16 floor
    return x.to(torch.bfloat16).contiguous()


@pytest.mark.parametrize("n_bits,rows,cols", [(8, 333, 7168), (10, 64, 2048), (3, 16, 256), (12, 16, 512)])
def test_logfmt_encode_matches_the_oracle(moe, orc, n_bits, rows, cols):
    x = _payload(rows, cols, rows + n_bits)
    ct = torch.uint8 if n_bits <= 8 else torch.int16
    codes = torch.empty(rows, cols, dtype=ct, device=DEV)
    lmin = torch.empty(rows, cols // 128, dtype=torch.float32, device=DEV)
    step = torch.empty_like(lmin)
    moe.moe_logfmt_encode(n_bits, x.view(torch.uint16), codes, lmin, step)
    torch.cuda.synchronize()
    ref = orc.logfmt_encode(to_host(x), n_bits)
    gl, gs = to_host(lmin), to_host(step)
    assert np.all(np.abs(gl - ref["lmin"]) <= 2e-6 * np.maximum(1, np.abs(ref["lmin"])))
    assert np.all(np.abs(gs - ref["step"]) <= 1e-5 * ref["step"])
    assert np.array_equal(gs == 0, ref["step"] == 0)
    gc = to_host(codes).astype(np.int64) & ((1 << n_bits) - 1)
    rc = ref["codes"].astype(np.int64)
    sure = ref["margin"] >= MARGIN
    assert np.array_equal(gc[sure], rc[sure]), np.argwhere((gc != rc) & sure)[:5]
    sign = 1 << (n_bits - 1)
    assert np.array_equal(gc & sign, rc & sign)
    assert np.all(np.abs((gc & (sign - 1)) - (rc & (sign - 1))) <= 1)
    assert sure.mean() > 0.99


@pytest.mark.parametrize("n_bits", [8, 10])
def test_logfmt_decode_matches_the_oracle(moe, orc, n_bits):
    rows, cols = 257, 7168
    x = to_host(_payload(rows, cols, 40 + n_bits))
    ref = orc.logfmt_encode(x, n_bits)                 # the oracle's codes and metadata...
    want = orc.round_bf16(orc.logfmt_decode(ref["codes"], ref["lmin"], ref["step"], n_bits))
    ct = np.uint8 if n_bits <= 8 else np.int16
    codes = torch.from_numpy(ref["codes"].astype(ct)).to(DEV)
    y = torch.empty(rows, cols, dtype=torch.bfloat16, device=DEV)
    moe.moe_logfmt_decode(n_bits, codes, torch.from_numpy(ref["lmin"]).to(DEV),
                          torch.from_numpy(ref["step"]).to(DEV), y.view(torch.uint16))   # ...decoded on the GPU
    torch.cuda.synchronize()
    got = to_host(y)
    diff = got != want
    # exp on the GPU is a few FP32 ulps off the oracle's: a BF16 rounding may land one unit off
    assert diff.mean() < 1e-3
    assert np.all(np.abs(got[diff].astype(np.int32) - want[diff].astype(np.int32)) <= 1)


def test_logfmt_round_trip_and_empty(moe):
    rows, cols, n_bits = 128, 7168, 8
    x = _payload(rows, cols, 99)
    codes = torch.empty(rows, cols, dtype=torch.uint8, device=DEV)
    lmin = torch.empty(rows, cols // 128, dtype=torch.float32, device=DEV)
    step = torch.empty_like(lmin)
    y = torch.empty_like(x)
    moe.moe_logfmt_encode(n_bits, x.view(torch.uint16), codes, lmin, step)
    moe.moe_logfmt_decode(n_bits, codes, lmin, step, y.view(torch.uint16))
    torch.cuda.synchronize()
    xf, yf = x.float().cpu().numpy().astype(np.float64), y.float().cpu().numpy().astype(np.float64)
    st = np.repeat(to_host(step), 128, 1).astype(np.float64)
    nz = (xf != 0) & (np.abs(xf) >= np.exp(np.repeat(to_host(lmin), 128, 1)))
    # a value on the grid's span decodes within half a gap (a relative e^Step - 1 at most)
    # plus the BF16 rounding of the decoded value
    rel = np.abs(yf - xf) / np.abs(np.where(nz, xf, 1))
    assert np.all(rel[nz] <= 0.5 * np.expm1(st[nz]) * 1.001 + 2 ** -8)
    assert np.array_equal(np.signbit(yf), np.signbit(xf))
    moe.moe_logfmt_encode(n_bits, x[:0].view(torch.uint16), codes[:0], lmin[:0], step[:0])
