"""Pins of the oracle's LogFMT-nBit codec (Insights into DeepSeek-V3 précis §3.2, LogFMT
communication compression) against what the passage fixes: the min / max of the log
magnitudes map to codes 1 and 2^(n-1) - 1, Step = (max - min) / (2^(n-1) - 2), zero is code 0,
values decode to exp(min + Step (K - 1)), rounding is nearest in linear space (unbiased, unlike
nearest in log space), and min is held above max - ln 2^32.  CPU only."""
import numpy as np
import pytest


def _tile(vals):
    x = np.zeros((1, 128), np.float32)
    x[0, :len(vals)] = vals
    return x


@pytest.mark.parametrize("n_bits", [8, 10])
def test_grid_points_get_their_own_codes(orc, n_bits):
    kmax = (1 << (n_bits - 1)) - 1
    lmin0, lmax0 = -3.0, 2.5
    step0 = (lmax0 - lmin0) / (kmax - 1)
    K = np.unique(np.linspace(1, kmax, 127).round().astype(int))
    vals = np.exp(lmin0 + step0 * (K - 1)).astype(np.float32)
    r = orc.logfmt_encode(_tile(vals), n_bits)
    # min and max of the tile are the first and last grid points: codes 1 and kmax
    assert abs(r["lmin"][0, 0] - np.float32(np.log(vals.min()))) <= 2e-7 * 3
    want_step = (np.log(np.float64(vals.max())) - np.log(np.float64(vals.min()))) / (kmax - 1)
    assert abs(r["step"][0, 0] - want_step) <= 1e-6 * want_step
    assert r["codes"][0, :len(K)].tolist() == K.tolist()
    assert not r["codes"][0, len(K):].any()          # the zero padding: code 0
    dec = orc.logfmt_decode(r["codes"], r["lmin"], r["step"], n_bits)
    assert np.allclose(dec[0, :len(K)], vals, rtol=2e-6, atol=0)
    assert not dec[0, len(K):].any()


def test_zero_and_sign(orc):
    x = _tile([1.0, -1.0, 0.5, -0.25, -0.0, 0.0, 4.0])
    r = orc.logfmt_encode(x, 8)
    c = r["codes"][0]
    assert c[4] == 0x80 and c[5] == 0 and c[7] == 0  # -0 keeps its sign bit; zeros are K = 0
    assert (c[1] & 0x80) and (c[3] & 0x80) and not (c[0] & 0x80)
    assert (c[1] & 0x7F) == (c[0] & 0x7F)            # magnitude code independent of the sign
    assert (c[6] & 0x7F) == 127 and (c[3] & 0x7F) == 1
    dec = orc.logfmt_decode(r["codes"], r["lmin"], r["step"], 8)[0]
    assert dec[1] < 0 and dec[3] < 0 and np.signbit(dec[4])
    assert np.isclose(dec[6], 4.0, rtol=1e-6) and np.isclose(dec[3], -0.25, rtol=1e-6)


def test_all_zero_tile_and_single_magnitude(orc):
    r = orc.logfmt_encode(np.zeros((2, 256), np.float32), 8)
    assert not r["codes"].any() and not r["lmin"].any() and not r["step"].any()
    r = orc.logfmt_encode(_tile([0.75, -0.75, 0.75]), 8)
    assert r["step"][0, 0] == 0 and r["codes"][0, :3].tolist() == [1, 0x81, 1]
    assert np.allclose(orc.logfmt_decode(r["codes"], r["lmin"], r["step"], 8)[0, :3], [0.75, -0.75, 0.75])


def test_rounding_is_nearest_in_linear_space(orc):
    # grid from the tile's own min 1 and max e^(126 * 0.05): d(K) = e^(0.05 (K - 1))
    n_bits, kmax = 8, 127
    lo_v, hi_v = np.float32(1.0), np.float32(np.exp(0.05 * (kmax - 1)))
    r0 = orc.logfmt_encode(_tile([lo_v, hi_v]), n_bits)
    lmin, step = float(r0["lmin"][0, 0]), float(r0["step"][0, 0])
    d = lambda K: np.exp(lmin + step * (K - 1))  # noqa: E731  (the decoder's grid)
    tests, want = [], []
    for K in (3, 40, 100):
        gm = np.sqrt(d(K) * d(K + 1))          # log-space midpoint: linear nearest is d(K)
        am = 0.5 * (d(K) + d(K + 1))           # linear-space midpoint
        for v, k in ((gm, K), (am * (1 + 1e-5), K + 1), (am * (1 - 1e-5), K)):
            tests.append(np.float32(v))
            want.append(k)
    r = orc.logfmt_encode(_tile([lo_v, hi_v] + tests), n_bits)
    assert r["lmin"][0, 0] == r0["lmin"][0, 0] and r["step"][0, 0] == r0["step"][0, 0]
    assert r["codes"][0, 2:2 + len(tests)].tolist() == want
    # below the first grid point: nearest of 0 and d(1)
    r = orc.logfmt_encode(_tile([lo_v, hi_v]), n_bits)
    assert r["codes"][0, 0] == 1


def test_min_is_held_above_max_minus_ln_2_pow_32(orc):
    x = _tile([1.0, 1e-12, 2.0e-10, 1.0e-10, 0.5])
    r = orc.logfmt_encode(x, 8)
    assert np.isclose(r["lmin"][0, 0], -32 * np.log(2.0), rtol=1e-7)
    d1 = 2.0 ** -32
    c = r["codes"][0]
    assert c[1] == 0                   # 1e-12 < d(1)/2: rounds to zero
    assert c[2] == 1                   # 2e-10 nearer d(1) = 2.3e-10 than 0
    assert c[3] == (0 if 1.0e-10 < d1 / 2 else 1)
    assert c[0] == 127


def test_linear_rounding_is_unbiased_and_log_rounding_is_not(orc):
    # many values spread uniformly over one gap [d(K), d(K+1)]: nearest-in-linear-space decodes
    # with a mean error of ~0; nearest-in-log-space (boundary at the geometric mean) would
    # round too many values up
    r0 = orc.logfmt_encode(_tile([1.0, np.exp(0.2 * 126)]), 8)
    lmin, step = float(r0["lmin"][0, 0]), float(r0["step"][0, 0])
    K = 60
    lo, hi = np.exp(lmin + step * (K - 1)), np.exp(lmin + step * K)
    vals = np.linspace(lo, hi, 126 * 40 + 2)[1:-1].astype(np.float32)
    errs = []
    for i in range(0, vals.size, 126):
        chunk = vals[i:i + 126]
        r = orc.logfmt_encode(_tile([1.0, np.float32(np.exp(0.2 * 126))] + chunk.tolist()), 8)
        assert r["lmin"][0, 0] == r0["lmin"][0, 0] and r["step"][0, 0] == r0["step"][0, 0]
        dec = orc.logfmt_decode(r["codes"], r["lmin"], r["step"], 8)[0, 2:2 + chunk.size]
        errs.append(dec.astype(np.float64) - chunk)
    e = np.concatenate(errs)
    gap = hi - lo
    assert abs(e.mean()) < 2e-3 * gap
    gm = np.sqrt(lo * hi)
    log_nearest = np.where(vals >= gm, hi, lo)
    assert (log_nearest - vals).mean() > 0.01 * gap   # ~(AM - GM) / gap = 2.5 % here


def test_round_trip_error_is_at_most_half_a_gap(orc):
    rng = np.random.default_rng(4)
    x = (rng.standard_normal((64, 1024)) * np.exp(rng.uniform(-4, 4, (64, 1))))
    x[3, :128] = 0
    x = x.astype(np.float32)
    r = orc.logfmt_encode(x, 8)
    dec = orc.logfmt_decode(r["codes"], r["lmin"], r["step"], 8).astype(np.float64)
    lm = np.repeat(r["lmin"], 128, 1).astype(np.float64)
    st = np.repeat(r["step"], 128, 1).astype(np.float64)
    a = np.abs(x.astype(np.float64))
    nz = a > 0
    # the gap around each value on the decoder's grid
    k = np.floor((np.log(np.where(nz, a, 1)) - lm) / np.where(st > 0, st, 1)) + 1
    lo = np.where(k >= 1, np.exp(lm + st * (k - 1)), 0)
    hi = np.exp(lm + st * k)
    inside = nz & (k >= 0) & (k < 127)
    assert np.all(np.abs(dec - x)[inside] <= 0.5 * (hi - lo)[inside] * (1 + 1e-6) + 1e-30)
    assert np.array_equal(np.signbit(dec[nz]), np.signbit(x[nz]))


def test_eight_bit_code_beats_e4m3_on_gaussian_tiles(orc):
    # the précis: at n = 8 LogFMT is more precise than E4M3 (here with the same 1x128 tiles and
    # the E4M3 quantiser's amax/448 scales)
    rng = np.random.default_rng(5)
    x = rng.standard_normal((256, 1024)).astype(np.float32)
    r = orc.logfmt_encode(x, 8)
    dec = orc.logfmt_decode(r["codes"], r["lmin"], r["step"], 8)
    q, s = orc.quant_1x128(x)
    e4 = orc.e4m3_table()[q] * np.repeat(s, 128, 1)
    rel = lambda y: np.mean(np.abs(y - x) / np.abs(x))  # noqa: E731
    assert rel(dec) < rel(e4)
