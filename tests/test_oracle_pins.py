"""Pins of the CPU oracle to facts outside itself (no GPU).

Each test checks the oracle against something it does not compute itself: the OCP OFP8
code table, library routines (torch's FP8/BF16 casts, numpy's stable argsort and float64
matmul, torch's silu), brute-force enumeration on tiny inputs, closed forms and
invariants stated on the pages:
  - DeepSeek-V3 co-design teardown (wsisp.com) §2.2 MoEGate listing, §2.3 dispatch skeleton,
    §5.1 blockwise FP8 GEMM sketch;
  - Insights into DeepSeek-V3 (Chinese précis) §3.1 (8 routed + 1 shared), §3.2
    (1x128 activation tiles, 128x128 weight blocks, FP32 accumulation).
"""
import itertools
import math
import os

import numpy as np
import pytest
import torch

HERE = os.path.dirname(os.path.abspath(__file__))


# ------------------------------------------------------------------ E4M3 / BF16 codecs

def _golden_e4m3():
    rows = []
    with open(os.path.join(HERE, "golden", "e4m3_ocp_codes.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                code, val = line.split()[:2]
                rows.append((int(code, 16), float(val)))
    return rows


def test_e4m3_table_matches_ocp_code_points(orc):
    table = orc.e4m3_table()
    for code, val in _golden_e4m3():
        if math.isnan(val):
            assert math.isnan(table[code]), hex(code)
        else:
            assert table[code] == val and math.copysign(1, table[code]) == math.copysign(1, val), hex(code)


def test_e4m3_table_matches_torch_decode_all_256_codes(orc):
    table = orc.e4m3_table()
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(table), nan)
    assert np.array_equal(table[~nan], ref[~nan])
    # the positive finite codes are strictly increasing (the encoder's search relies on it)
    assert np.all(np.diff(table[:127]) > 0)


def _e4m3_probe_values():
    t = np.sort(np.unique(np.abs(torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn)
                                 .to(torch.float32).numpy())))
    t = t[np.isfinite(t)]
    mids = ((t[:-1].astype(np.float64) + t[1:]) / 2).astype(np.float32)  # exact midpoints
    near = np.concatenate([np.nextafter(mids, np.float32(0)), np.nextafter(mids, np.float32(1e9)),
                           mids, t])
    rng = np.random.default_rng(1)
    rand = np.concatenate([rng.uniform(0, 448, 4000), np.exp(rng.uniform(-16, 6.1, 4000))])
    v = np.concatenate([near, rand.astype(np.float32)])
    v = v[v <= 448].astype(np.float32)
    return np.concatenate([v, -v])


def test_e4m3_encode_matches_torch_round_to_nearest_even(orc):
    v = _e4m3_probe_values()
    ours = orc.f32_to_e4m3(v)
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    bad = np.nonzero(ours != ref)[0]
    assert bad.size == 0, [(float(v[i]), hex(ours[i]), hex(ref[i])) for i in bad[:10]]


def test_e4m3_encode_ties_go_to_even_code(orc):
    table = orc.e4m3_table()
    for c in range(0, 126):
        mid = np.float32((table[c] + table[c + 1]) / 2)
        assert float(mid) == (table[c] + table[c + 1]) / 2  # midpoint exact in FP32
        want = c if c % 2 == 0 else c + 1
        assert orc.f32_to_e4m3(np.array([mid]))[0] == want, c


def test_e4m3_encode_saturates(orc):
    v = np.array([448.0, 448.5, 463.99, 464.0, 480.0, 1e6, np.inf, -450.0, -np.inf, np.nan],
                 np.float32)
    got = orc.f32_to_e4m3(v)
    assert list(got[:7]) == [0x7E] * 7
    assert list(got[7:9]) == [0xFE] * 2
    assert got[9] == 0x7F


def test_bf16_rounding_matches_torch(orc):
    rng = np.random.default_rng(2)
    base = (rng.standard_normal(3000) * 10.0 ** rng.integers(-5, 5, 3000)).astype(np.float32)
    u = base.view(np.uint32)
    ties = ((u & 0xFFFF0000) | 0x8000).view(np.float32)  # exact halfway cases
    v = np.concatenate([base, ties, np.float32([0.0, -0.0, 3.3895314e38, 1e-40])])
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.uint16).numpy()
    assert np.array_equal(orc.f32_to_bf16(v), ref)
    assert np.array_equal(orc.round_bf16(v), ref)
    assert np.array_equal(orc.bf16_to_f32(ref), torch.from_numpy(ref).view(torch.bfloat16).float().numpy())


# ------------------------------------------------------------------ 1x128 / 128x128 quantisation

def test_quant_1x128_tile_properties(orc):
    rng = np.random.default_rng(3)
    x = rng.standard_normal((5, 512)).astype(np.float32)
    x[1, 128:256] = 0.0                         # all-zero tile
    x[2, 256:384] = 0.0
    x[2, 300] = -3.5                            # single non-zero
    x[3, :128] *= np.float32(1e-3)              # small tile
    x[4, 384:] = np.float32(2.0) ** rng.integers(-20, 20, 128).astype(np.float32)  # wide range
    q, s = orc.quant_1x128(x)
    table = orc.e4m3_table()
    for r in range(x.shape[0]):
        for b in range(4):
            tile = x[r, b * 128:(b + 1) * 128]
            amax = np.float32(np.max(np.abs(tile)))
            qt = q[r, b * 128:(b + 1) * 128]
            if amax == 0:
                assert s[r, b] == 1.0 and not qt.any()
                continue
            assert s[r, b] == np.float32(amax / np.float32(448.0))
            # the largest magnitude maps to the largest code
            k = int(np.argmax(np.abs(tile)))
            assert qt[k] == (0xFE if tile[k] < 0 else 0x7E)
            # every code is the library's nearest-even E4M3 of the FP32 product v * (448/amax)
            mul = np.float32(np.float32(448.0) / amax)
            ref = torch.from_numpy((tile * mul).astype(np.float32)).clamp(-448, 448) \
                .to(torch.float8_e4m3fn).view(torch.uint8).numpy()
            assert np.array_equal(qt, ref)
            # dequantised error within half a code step of the scaled value
            dq = table[qt] * np.float64(s[r, b])
            step = np.array([_e4m3_gap(table, abs(float(v) * float(mul))) for v in tile])
            assert np.all(np.abs(dq - tile) <= 0.5 * step * float(s[r, b]) * (1 + 1e-6) + 1e-30)


def _e4m3_gap(table, a):
    pos = table[:127]
    i = np.searchsorted(pos, a, side="right") - 1
    i = min(max(i, 0), 125)
    return pos[i + 1] - pos[i]


def test_quant_128x128_block_layout(orc):
    rng = np.random.default_rng(4)
    n, R, C = 2, 256, 384
    w = rng.standard_normal((n, R, C)).astype(np.float32)
    # give every block its own magnitude so a transposed or shifted block index shows
    for m in range(n):
        for i in range(R // 128):
            for j in range(C // 128):
                w[m, i * 128:(i + 1) * 128, j * 128:(j + 1) * 128] *= np.float32(2.0 ** (i + 3 * j + 7 * m - 6))
    w[1, :128, 128:256] = 0.0
    q, s = orc.quant_128x128(w)
    for m in range(n):
        for i in range(R // 128):
            for j in range(C // 128):
                blk = w[m, i * 128:(i + 1) * 128, j * 128:(j + 1) * 128]
                amax = np.float32(np.abs(blk).max())
                qb = q[m, i * 128:(i + 1) * 128, j * 128:(j + 1) * 128]
                if amax == 0:
                    assert s[m, i, j] == 1.0 and not qb.any()
                    continue
                assert s[m, i, j] == np.float32(amax / np.float32(448.0))
                mul = np.float32(np.float32(448.0) / amax)
                ref = torch.from_numpy(blk * mul).clamp(-448, 448).to(torch.float8_e4m3fn) \
                    .view(torch.uint8).numpy()
                assert np.array_equal(qb, ref)
    # BF16 input path reads the same values as the FP32 path
    wb = torch.from_numpy(w).to(torch.bfloat16)
    qb16, sb16 = orc.quant_128x128(wb.view(torch.uint16).numpy())
    q32, s32 = orc.quant_128x128(wb.float().numpy())
    assert np.array_equal(qb16, q32) and np.array_equal(sb16, s32)


# ------------------------------------------------------------------ gate

def _rand_gate_case(rng, T, H, E, bias_scale=0.1):
    x = rng.standard_normal((T, H)).astype(np.float32)
    Wg = (rng.standard_normal((E, H)) * 0.3).astype(np.float32)
    b = rng.uniform(-bias_scale, bias_scale, E).astype(np.float32)
    return x, Wg, b


def test_gate_logits_and_sigmoid_against_float64_matmul(orc):
    rng = np.random.default_rng(5)
    x, Wg, b = _rand_gate_case(rng, 40, 96, 16)
    g = orc.gate(x, Wg, b, 4, 2, 2, 1.0, want_scores=True)
    logits = (x.astype(np.float64) @ Wg.astype(np.float64).T).astype(np.float32)
    ref = torch.sigmoid(torch.from_numpy(logits).double()).float().numpy()
    assert np.array_equal(g["scores"], ref)


def test_gate_sigmoid_closed_forms(orc):
    # logit 0 -> 0.5; logit ln 3 -> 0.75 (single one-hot feature times a chosen weight)
    H, E = 4, 8
    x = np.zeros((1, H), np.float32)
    x[0, 0] = 1.0
    Wg = np.zeros((E, H), np.float32)
    Wg[3, 0] = np.float32(math.log(3.0))
    g = orc.gate(x, Wg, np.zeros(E, np.float32), 4, 4, 1, 2.0, want_scores=True)
    s = g["scores"][0]
    assert s[0] == 0.5 and abs(s[3] - 0.75) < 1e-7
    assert g["topk_idx"][0, 0] == 3
    # top_k = 1: no renormalisation; weight = rsf * sigmoid(logit)
    assert g["topk_w"][0, 0] == np.float32(s[3] * np.float32(2.0))


def _brute_force_selection(c, G, TG, K):
    """Kept groups = the TG-subset with the largest total group score, where a group's
    score is its best pair sum; chosen experts = the K-subset of allowed experts with the
    largest sum of selection scores."""
    E = c.size
    gsz = E // G
    gscore = []
    for g in range(G):
        vals = c[g * gsz:(g + 1) * gsz]
        gscore.append(max(np.float32(vals[i] + vals[j]) for i, j in itertools.combinations(range(gsz), 2)))
    best_groups = max(itertools.combinations(range(G), TG),
                      key=lambda S: sum(float(gscore[g]) for g in S))
    allowed = [e for e in range(E) if e // gsz in best_groups]
    best = max(itertools.combinations(allowed, K), key=lambda S: sum(float(c[e]) for e in S))
    return set(best)


@pytest.mark.parametrize("E,G,TG,K", [(16, 4, 2, 2), (8, 4, 2, 3), (12, 3, 2, 4), (16, 4, 3, 1),
                                      (16, 8, 4, 5), (6, 2, 1, 3)])
def test_gate_selection_brute_force(orc, E, G, TG, K):
    rng = np.random.default_rng(100 + E * 10 + K)
    x, Wg, b = _rand_gate_case(rng, 60, 32, E)
    g = orc.gate(x, Wg, b, G, TG, K, 1.0, want_scores=True)
    c = (g["scores"] + b[None, :]).astype(np.float32)
    for t in range(x.shape[0]):
        assert set(g["topk_idx"][t].tolist()) == _brute_force_selection(c[t], G, TG, K), t
        # slots in descending selection score
        ct = c[t][g["topk_idx"][t]]
        assert np.all(np.diff(ct) <= 0)


def test_gate_ties_go_to_lower_index(orc):
    # all scores equal: keep groups 0..TG-1, experts in ascending index
    T, H, E = 3, 8, 16
    x = np.ones((T, H), np.float32)
    Wg = np.zeros((E, H), np.float32)
    g = orc.gate(x, Wg, np.zeros(E, np.float32), 4, 2, 3, 1.0)
    assert g["topk_idx"].tolist() == [[0, 1, 2]] * T
    assert np.all(g["margin"] == 0)


def _margin_case(orc, bias_units, G, TG, K):
    """Zero logits give every score exactly 1/2, so the selection scores are 1/2 + b; with b
    a multiple of u = 2^-20 every selection score, group score and margin below is exact."""
    E = len(bias_units)
    u = 2.0 ** -20
    b = (np.asarray(bias_units, np.float64) * u).astype(np.float32)
    x = np.zeros((2, 32), np.float32)
    Wg = np.zeros((E, 32), np.float32)
    return orc.gate(x, Wg, b, G, TG, K, 1.0), u


def test_gate_margin_is_the_smaller_of_the_two_cuts(orc):
    # groups of 4; the margin is min(TG-th kept group score - best dropped group score,
    # K-th chosen selection score - best unchosen candidate in the kept groups)
    # group scores (top-2 sums, in units over 1): g0 19, g1 14, g2 13, g3 0 -> group cut 1
    # kept experts by score: 10, 9, 8, then 6 -> expert cut (K = 3) 2
    g, u = _margin_case(orc, [10, 9, 0, 0, 8, 6, 0, 0, 7, 6, 0, 0, 0, 0, 0, 0], 4, 2, 3)
    assert g["topk_idx"][0].tolist() == [0, 1, 4]
    assert np.all(g["margin"] == np.float32(u))
    # a wider group cut (g2 9): now the expert cut, 2 units, is the smaller
    g, u = _margin_case(orc, [10, 9, 0, 0, 8, 6, 0, 0, 5, 4, 0, 0, 0, 0, 0, 0], 4, 2, 3)
    assert np.all(g["margin"] == np.float32(2 * u))
    # every group kept: no group cut, the expert cut alone (top-4: 10 9 8 7, next 6 -> 1)
    g, u = _margin_case(orc, [10, 9, 0, 0, 8, 6, 0, 0, 7, 3, 0, 0, 0, 0, 0, 0], 4, 4, 4)
    assert g["topk_idx"][0].tolist() == [0, 1, 4, 8]
    assert np.all(g["margin"] == np.float32(u))
    # K takes every expert of the kept groups: no expert cut, the group cut alone (19 - 14 = 5)
    g, u = _margin_case(orc, [10, 9, 1, 0, 8, 6, 0, 0, 7, 7, 0, 0, 0, 0, 0, 0], 4, 1, 4)
    assert sorted(g["topk_idx"][0].tolist()) == [0, 1, 2, 3]
    assert np.all(g["margin"] == np.float32(5 * u))
    # an exact tie at the expert cut (8 and 8) gives margin 0; the lower index is chosen
    g, u = _margin_case(orc, [10, 9, 0, 0, 8, 0, 0, 0, 8, 6, 0, 0, 0, 0, 0, 0], 4, 3, 3)
    assert g["topk_idx"][0].tolist() == [0, 1, 4]
    assert np.all(g["margin"] == 0)
    # an exact tie at the group cut (14 and 14, top-1 group... g1 and g2 tie for the 2nd)
    g, u = _margin_case(orc, [10, 9, 0, 0, 8, 6, 0, 0, 7, 7, 0, 0, 0, 0, 0, 0], 4, 2, 2)
    assert g["topk_idx"][0].tolist() == [0, 1]
    assert np.all(g["margin"] == 0)


def test_gate_masked_experts_never_chosen_even_with_negative_scores(orc):
    # every selection score negative: the kept groups still bound the choice
    rng = np.random.default_rng(6)
    x, Wg, _ = _rand_gate_case(rng, 30, 16, 16)
    b = np.full(16, -3.0, np.float32)
    b[:4] -= 1.0  # group 0 is worst
    g = orc.gate(x, Wg, b, 4, 2, 4, 1.0, want_scores=True)
    c = g["scores"] + b
    for t in range(30):
        assert set(g["topk_idx"][t].tolist()) == _brute_force_selection(c[t].astype(np.float32), 4, 2, 4)


def test_gate_weights_normalised_and_scaled(orc):
    rng = np.random.default_rng(7)
    x, Wg, b = _rand_gate_case(rng, 50, 24, 16)
    for K, rsf in [(2, 1.0), (4, 2.5), (6, 0.5)]:
        g = orc.gate(x, Wg, b, 4, 3, K, rsf)
        assert np.allclose(g["topk_w"].sum(1, dtype=np.float64), rsf, rtol=2e-6, atol=0)


def test_gate_bias_changes_selection_but_not_weight_values(orc):
    rng = np.random.default_rng(8)
    x, Wg, _ = _rand_gate_case(rng, 200, 24, 16)
    zero = np.zeros(16, np.float32)
    big = rng.uniform(-0.3, 0.3, 16).astype(np.float32)
    for K in (1, 3):
        g0 = orc.gate(x, Wg, zero, 4, 2, K, 1.5, want_scores=True)
        g1 = orc.gate(x, Wg, big, 4, 2, K, 1.5, want_scores=True)
        assert np.array_equal(g0["scores"], g1["scores"])  # the bias never enters the scores
        changed = np.any(np.sort(g0["topk_idx"], 1) != np.sort(g1["topk_idx"], 1), axis=1)
        assert changed.any() and not changed.all()
        same = ~changed
        o0 = np.argsort(g0["topk_idx"], 1)
        o1 = np.argsort(g1["topk_idx"], 1)
        w0 = np.take_along_axis(g0["topk_w"], o0, 1)
        w1 = np.take_along_axis(g1["topk_w"], o1, 1)
        # same selected set -> the same weights, whatever the bias (bit-identical when the
        # slot order agrees too; otherwise the normalising sum runs in another order)
        same_order = np.all(g0["topk_idx"] == g1["topk_idx"], axis=1)
        assert np.array_equal(g0["topk_w"][same_order], g1["topk_w"][same_order])
        assert np.allclose(w0[same], w1[same], rtol=3e-7, atol=0)
        # weights follow the un-biased scores of the chosen experts
        s_sel = np.take_along_axis(g1["scores"], g1["topk_idx"], 1)
        if K == 1:
            assert np.array_equal(g1["topk_w"][:, 0], s_sel[:, 0] * np.float32(1.5))
        else:
            ratio = g1["topk_w"] / s_sel
            assert np.allclose(ratio, ratio[:, :1], rtol=1e-6)


# ------------------------------------------------------------------ permutation, bias update

def test_permute_matches_stable_argsort(orc):
    rng = np.random.default_rng(9)
    T, E, K = 300, 16, 4
    idx = np.stack([rng.choice(E, K, replace=False) for _ in range(T)]).astype(np.int32)
    idx[5] = [0, 1, 2, 3]
    for has_shared in (0, 1):
        p = orc.permute(idx, E, has_shared)
        flat = idx.ravel()
        order = np.argsort(flat, kind="stable")
        assert np.array_equal(p["perm_tok"][:T * K], order // K)
        assert np.array_equal(p["counts"], np.bincount(flat, minlength=E))
        assert np.array_equal(p["offs"][:E + 1], np.concatenate([[0], np.cumsum(p["counts"])]))
        rows = p["row_of"].ravel()
        assert np.array_equal(np.sort(rows), np.arange(T * K))
        assert np.array_equal(p["perm_tok"][rows], np.repeat(np.arange(T), K))
        for e in range(E):  # every row lies in its expert's range
            r = p["row_of"][idx == e]
            assert np.all((r >= p["offs"][e]) & (r < p["offs"][e + 1]))
        if has_shared:
            assert p["offs"][E + 1] == T * K + T
            assert np.array_equal(p["perm_tok"][T * K:], np.arange(T))


def test_permute_empty_and_full_experts(orc):
    T, E, K = 50, 8, 2
    idx = np.tile(np.array([[6, 2]], np.int32), (T, 1))
    p = orc.permute(idx, E, 0)
    assert p["counts"].tolist() == [0, 0, T, 0, 0, 0, T, 0]
    assert p["offs"].tolist() == [0, 0, 0, T, T, T, T, 2 * T, 2 * T]
    assert np.array_equal(p["row_of"][:, 0], np.arange(T) + T)
    assert np.array_equal(p["row_of"][:, 1], np.arange(T))


def test_permute_drops_ids_outside_range(orc):
    # the library's contract for ids the gate never produces: such a slot counts for no
    # expert and gets no row (row_of -1); the valid slots keep the stable expert-major order
    # in rows [0, V) and the rows [V, T*K) are unclaimed (perm_tok -1), the shared group
    # still starting at T*K
    rng = np.random.default_rng(21)
    T, E, K = 97, 12, 3
    idx = np.stack([rng.choice(E, K, replace=False) for _ in range(T)]).astype(np.int32)
    idx[4, 1] = -1
    idx[10, 0] = E
    idx[50, 2] = 1 << 20
    idx[96] = [-5, -6, -7]
    for has_shared in (0, 1):
        p = orc.permute(idx, E, has_shared)
        flat = idx.ravel()
        ok = (flat >= 0) & (flat < E)
        V = int(ok.sum())
        pos = np.nonzero(ok)[0]
        order = pos[np.argsort(flat[ok], kind="stable")]
        assert np.array_equal(p["perm_tok"][:V], order // K)
        assert np.all(p["perm_tok"][V:T * K] == -1)
        assert np.array_equal(p["counts"], np.bincount(flat[ok], minlength=E))
        assert np.array_equal(p["offs"][:E], np.concatenate([[0], np.cumsum(p["counts"])[:-1]]))
        assert p["offs"][E] == T * K
        rows = p["row_of"].ravel()
        assert np.all(rows[~ok] == -1)
        assert np.array_equal(np.sort(rows[ok]), np.arange(V))
        assert np.array_equal(p["perm_tok"][rows[ok]], pos // K)
        if has_shared:
            assert p["offs"][E + 1] == T * K + T
            assert np.array_equal(p["perm_tok"][T * K:], np.arange(T))


def test_bias_update_hand_examples(orc):
    # T*K/E = 4*2/4 = 2: loads below, at and above the mean
    b = np.array([0.5, 0.0, -0.25, 1.0], np.float32)
    counts = np.array([1, 2, 5, 0], np.int32)
    nb = orc.bias_update(counts, b, T=4, top_k=2)
    assert nb.tolist() == [np.float32(0.5) + np.float32(1e-3), 0.0,
                           np.float32(-0.25) - np.float32(1e-3), np.float32(1.0) + np.float32(1e-3)]
    # non-integer mean (T*K/E = 7/3): compare in integers, no rounding trap
    nb = orc.bias_update(np.array([2, 3, 2], np.int32), np.zeros(3, np.float32), T=7, top_k=1)
    assert nb.tolist() == [np.float32(1e-3), np.float32(-1e-3), np.float32(1e-3)]


# ------------------------------------------------------------------ experts

def _tiny_fp8_expert_case(rng, n, H, I, nE):
    x = rng.standard_normal((n, H)).astype(np.float32)
    W13 = (rng.standard_normal((nE, 2 * I, H)) * 0.05).astype(np.float32)
    W2 = (rng.standard_normal((nE, H, I)) * 0.05).astype(np.float32)
    return x, W13, W2


def _dequant(table, q, s, rb, cb):
    v = table[q]
    return v * np.repeat(np.repeat(s.astype(np.float64), rb, axis=-2), cb, axis=-1)


def test_ffn_fp8_against_dense_float64_matmul(orc):
    rng = np.random.default_rng(10)
    n, H, I, nE = 6, 384, 256, 3
    x, W13, W2 = _tiny_fp8_expert_case(rng, n, H, I, nE)
    xq, xs = orc.quant_1x128(x)
    W13q, W13s = orc.quant_128x128(W13)
    W2q, W2s = orc.quant_128x128(W2)
    row_e = np.array([0, 1, 2, 2, 1, 0], np.int32)
    y, aux = orc.ffn_fp8(xq, xs, row_e, W13q, W13s, W2q, W2s, want_h=True)
    t = orc.e4m3_table()
    A = _dequant(t, xq, xs, 1, 128)
    for r in range(n):
        e = row_e[r]
        Wd = _dequant(t, W13q[e], W13s[e], 128, 128)
        gu = (A[r] @ Wd.T).astype(np.float32)
        assert np.array_equal(aux["gu"][r], gu), r
        # silu through the library routine, then the FP32 product
        h = (torch.nn.functional.silu(torch.from_numpy(gu[:I]).double()).numpy()
             * gu[I:].astype(np.float64)).astype(np.float32)
        assert np.array_equal(aux["h"][r], h)
        hq, hs = orc.quant_1x128(h[None])
        assert np.array_equal(aux["hq"][r], hq[0]) and np.array_equal(aux["hs"][r], hs[0])
        Hd = _dequant(t, hq, hs, 1, 128)[0]
        W2d = _dequant(t, W2q[e], W2s[e], 128, 128)
        yref = torch.from_numpy((W2d @ Hd).astype(np.float32)).to(torch.bfloat16).view(torch.uint16).numpy()
        assert np.array_equal(y[r], yref)


def test_ffn_fp8_single_block_by_hand(orc):
    # H = I = 128: one block per operand.  x = 1 everywhere -> codes 448, scale fl(1/448).
    # gate row j = 0.5 at k = j, up row j = 2.0 at k = j: each block's amax maps to code 448,
    # so g_j = 448*448*fl(1/448)*fl(0.5/448) and u_j = 448*448*fl(1/448)*fl(2/448).
    H = I = 128
    x = np.ones((1, H), np.float32)
    W13 = np.zeros((1, 2 * I, H), np.float32)
    W2 = np.zeros((1, H, I), np.float32)
    for j in range(I):
        W13[0, j, j] = 0.5
        W13[0, I + j, j] = 2.0
        W2[0, j, j] = 1.0
    xq, xs = orc.quant_1x128(x)
    assert xs[0, 0] == np.float32(1.0 / 448.0) and np.all(xq == 0x7E)
    qw = orc.quantize_weights(W13, W2)
    assert qw[1].ravel().tolist() == [np.float32(0.5 / 448), np.float32(2.0 / 448)]
    y, aux = orc.ffn_fp8(xq, xs, np.zeros(1, np.int32), *qw, want_h=True)
    sa = float(np.float32(1.0 / 448.0))
    g = np.float32(448.0 * 448.0 * sa * float(np.float32(0.5 / 448)))
    u = np.float32(448.0 * 448.0 * sa * float(np.float32(2.0 / 448)))
    assert np.all(aux["gu"][0, :I] == g) and np.all(aux["gu"][0, I:] == u)
    silu = float(g) / (1 + math.exp(-float(g)))
    assert np.all(aux["h"][0] == np.float32(silu * float(u)))
    # h is constant -> every code is 448; W2 = identity -> y_j = h_j up to the scales and BF16
    assert np.all(aux["hq"][0] == 0x7E)
    yf = orc.bf16_to_f32(y[0])
    assert np.allclose(yf, aux["h"][0], rtol=2 ** -8)


def test_ffn_zero_weight_expert_contributes_nothing(orc):
    rng = np.random.default_rng(11)
    n, H, I, nE = 4, 256, 128, 2
    x, W13, W2 = _tiny_fp8_expert_case(rng, n, H, I, nE)
    W2[1] = 0.0
    xq, xs = orc.quant_1x128(x)
    y = orc.ffn_fp8(xq, xs, np.array([1, 1, 0, 1], np.int32), *orc.quantize_weights(W13, W2))
    assert not y[[0, 1, 3]].any() and y[2].any()
    yf = orc.ffn_f32(x, np.array([1, 0, 1, 1], np.int32), W13, W2)
    assert not yf[[0, 2, 3]].any() and yf[1].any()


def test_ffn_f32_against_float64_matmul(orc):
    rng = np.random.default_rng(12)
    n, H, I, nE = 5, 64, 32, 2
    x, W13, W2 = _tiny_fp8_expert_case(rng, n, H, I, nE)
    row_e = np.array([1, 0, 1, 0, 0], np.int32)
    y, h = orc.ffn_f32(x, row_e, W13, W2, want_h=True)
    for r in range(n):
        gu = (x[r].astype(np.float64) @ W13[row_e[r]].astype(np.float64).T).astype(np.float32)
        hr = (torch.nn.functional.silu(torch.from_numpy(gu[:I]).double()).numpy() * gu[I:]).astype(np.float32)
        assert np.array_equal(h[r], hr)
        assert np.array_equal(y[r], (W2[row_e[r]].astype(np.float64) @ hr.astype(np.float64)).astype(np.float32))


# ------------------------------------------------------------------ combine, whole layer

def test_combine_closed_forms(orc):
    yk = np.array([[[1.0, 2.0, -4.0], [8.0, 0.5, 3.0]]], np.float32)  # [1, K=2, H=3]
    w = np.array([[0.25, 0.75]], np.float32)
    ysh = np.array([[1.0, 1.0, 1.0]], np.float32)
    acc = orc.combine(yk, w, ysh)
    assert acc.tolist() == [[0.25 + 6.0 + 1.0, 0.5 + 0.375 + 1.0, -1.0 + 2.25 + 1.0]]
    assert orc.combine(yk[:, :1], np.ones((1, 1), np.float32)).tolist() == [[1.0, 2.0, -4.0]]
    yb = torch.from_numpy(yk).to(torch.bfloat16).view(torch.uint16).numpy()
    sb = torch.from_numpy(ysh).to(torch.bfloat16).view(torch.uint16).numpy()
    assert np.array_equal(orc.combine(yb, w, sb), acc)


def _tiny_layer(rng, mode):
    cfg = dict(hidden=256, inter=128, n_experts=16, n_group=4, topk_group=2, top_k=2,
               routed_scaling_factor=1.0, has_shared=1, mode=mode)
    T = 24
    x = rng.standard_normal((T, 256)).astype(np.float32)
    Wg = (rng.standard_normal((16, 256)) * 0.02).astype(np.float32)
    b = rng.uniform(-0.1, 0.1, 16).astype(np.float32)
    W13 = (rng.standard_normal((17, 256, 256)) * 0.02).astype(np.float32)
    W2 = (rng.standard_normal((17, 256, 128)) * 0.02).astype(np.float32)
    return cfg, x, Wg, b, W13, W2


@pytest.mark.parametrize("mode", ["fp32", "fp8", "fp8_pow2"])
def test_forward_sample_is_exact_and_shared_only_when_routed_zero(orc, mode):
    rng = np.random.default_rng(13)
    cfg, x, Wg, b, W13, W2 = _tiny_layer(rng, mode)
    full = orc.forward(cfg, x, Wg, b, W13, W2)
    samp = np.array([3, 7, 20])
    part = orc.forward(cfg, x, Wg, b, W13, W2, sample=samp)
    assert np.array_equal(part["y"], full["y"][samp])
    # zero every routed down-projection: the layer output is the shared expert alone
    W2z = W2.copy()
    W2z[:16] = 0.0
    z = orc.forward(cfg, x, Wg, b, W13, W2z)
    if mode == "fp32":
        sh = orc.ffn_f32(x, np.full(x.shape[0], 16, np.int32), W13, W2)
        assert np.array_equal(z["y"], sh)
    else:
        pow2 = mode == "fp8_pow2"
        xq, xs = orc.quant_1x128(x, pow2)
        sh = orc.ffn_fp8(xq, xs, np.full(x.shape[0], 16, np.int32), *orc.quantize_weights(W13, W2, pow2),
                         pow2=pow2)
        assert np.array_equal(z["y"], sh)


def test_forward_top1_weight_is_scaled_score(orc):
    rng = np.random.default_rng(14)
    cfg, x, Wg, b, W13, W2 = _tiny_layer(rng, "fp32")
    cfg = dict(cfg, top_k=1, routed_scaling_factor=2.5)
    out = orc.forward(cfg, x, Wg, b, W13, W2)
    g = orc.gate(x, Wg, b, 4, 2, 1, 2.5, want_scores=True)
    s = np.take_along_axis(g["scores"], g["topk_idx"], 1)[:, 0]
    assert np.array_equal(out["topk_w"][:, 0], s * np.float32(2.5))


# ------------------------------------------------------------------ power-of-two scales
# Insights into DeepSeek-V3 (précis) §3.2 recommends tensor cores that take the scaling
# factors natively (Blackwell's microscaling), whose scales are powers of two.  The oracle's
# power-of-two mode takes the smallest power of two s with 448*s >= amax, clamped to
# 2^-127 .. 2^127, and encodes v * 2^-e.

def _check_pow2_tile(tile, codes, scale, table):
    amax = float(np.max(np.abs(tile)))
    if amax == 0:
        assert scale == 1.0 and not codes.any()
        return
    m, e2 = np.frexp(np.float64(scale))
    assert m == 0.5, scale                      # an exact power of two
    e = int(e2) - 1
    assert -127 <= e <= 127
    assert 448.0 * 2.0 ** e >= amax             # covers the tile: nothing saturates
    if e > -127:
        assert 448.0 * 2.0 ** (e - 1) < amax    # and is the smallest such power
        assert amax * 2.0 ** -e > 224.0         # so amax lands in the top binade of E4M3
    scaled = tile.astype(np.float64) * 2.0 ** -e  # exact
    assert np.max(np.abs(scaled)) <= 448.0
    ref = torch.from_numpy(scaled.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(codes, ref)
    # dequantised error within half a code step
    dq = table[codes] * np.float64(scale)
    step = np.array([_e4m3_gap(table, abs(float(v))) for v in scaled]) * np.float64(scale)
    assert np.all(np.abs(dq - tile) <= 0.5 * step * (1 + 1e-12) + 1e-300)


def test_pow2_quant_1x128_scales_and_codes(orc):
    rng = np.random.default_rng(21)
    x = rng.standard_normal((7, 512)).astype(np.float32)
    x[0, :128] *= np.float32(1e-3)
    x[1, 128:256] = 0.0                                            # all-zero tile
    x[2, :128] = np.clip(x[2, :128], -1, 1)
    x[2, 5] = np.float32(448 * 2.0 ** -3)                          # amax exactly 448 * 2^-3
    x[3, :128] = np.clip(x[3, :128], -1, 1)
    x[3, 7] = np.nextafter(np.float32(448 * 2.0 ** -2), np.float32(np.inf))  # just above 448 * 2^-2
    x[4, 256:384] = np.float32(2.0) ** rng.integers(-20, 20, 128).astype(np.float32)
    x[5, 384:] *= np.float32(1e-37)                                # exponent clamped at -127
    x[6, :128] = np.float32(-448 * 2.0 ** 5)                       # constant negative tile
    q, s = orc.quant_1x128(x, pow2=True)
    table = orc.e4m3_table()
    for r in range(x.shape[0]):
        for b in range(4):
            _check_pow2_tile(x[r, b * 128:(b + 1) * 128], q[r, b * 128:(b + 1) * 128], float(s[r, b]), table)
    assert s[2, 0] == np.float32(2.0 ** -3) and q[2, 5] == 0x7E     # amax -> code 448
    assert s[3, 0] == np.float32(2.0 ** -1)
    assert s[5, 3] == np.float32(2.0 ** -127)
    assert s[6, 0] == np.float32(2.0 ** 5) and np.all(q[6, :128] == 0xFE)
    # BF16 input reads the same values as the FP32 path
    xb = torch.from_numpy(x).to(torch.bfloat16)
    qb, sb = orc.quant_1x128(xb.view(torch.uint16).numpy(), pow2=True)
    qf, sf = orc.quant_1x128(xb.float().numpy(), pow2=True)
    assert np.array_equal(qb, qf) and np.array_equal(sb, sf)


def test_pow2_quant_128x128_block_layout(orc):
    rng = np.random.default_rng(22)
    n, R, C = 2, 256, 384
    w = rng.standard_normal((n, R, C)).astype(np.float32)
    # every block its own magnitude (not a power of two apart), so a transposed or shifted
    # block index shows in the scales
    for m in range(n):
        for i in range(R // 128):
            for j in range(C // 128):
                w[m, i * 128:(i + 1) * 128, j * 128:(j + 1) * 128] *= np.float32(3.0 ** (i + 2 * j + 5 * m - 6))
    w[1, :128, 128:256] = 0.0
    q, s = orc.quant_128x128(w, pow2=True)
    table = orc.e4m3_table()
    for m in range(n):
        for i in range(R // 128):
            for j in range(C // 128):
                blk = w[m, i * 128:(i + 1) * 128, j * 128:(j + 1) * 128]
                qb = q[m, i * 128:(i + 1) * 128, j * 128:(j + 1) * 128]
                sc = float(s[m, i, j])
                for r in range(0, 128, 37):      # rows of the block share its one scale
                    amax = float(np.abs(blk).max())
                    if amax == 0:
                        assert sc == 1.0 and not qb.any()
                        continue
                    e = int(np.frexp(np.float64(sc))[1]) - 1
                    assert 448.0 * 2.0 ** e >= amax > 448.0 * 2.0 ** (e - 1)
                    scaled = blk[r].astype(np.float64) * 2.0 ** -e
                    ref = torch.from_numpy(scaled.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
                    assert np.array_equal(qb[r], ref)
    assert len({float(v) for v in s.ravel()}) > 6


def test_pow2_ffn_against_dense_float64_matmul(orc):
    # the blockwise sum is the same for either kind of scale: g, u and y still equal the
    # float64 matmul of the dequantised operands, and h is re-quantised with power-of-two scales
    rng = np.random.default_rng(23)
    n, H, I, nE = 5, 384, 256, 2
    x, W13, W2 = _tiny_fp8_expert_case(rng, n, H, I, nE)
    xq, xs = orc.quant_1x128(x, pow2=True)
    W13q, W13s, W2q, W2s = orc.quantize_weights(W13, W2, pow2=True)
    row_e = np.array([0, 1, 1, 0, 1], np.int32)
    y, aux = orc.ffn_fp8(xq, xs, row_e, W13q, W13s, W2q, W2s, want_h=True, pow2=True)
    t = orc.e4m3_table()
    A = _dequant(t, xq, xs, 1, 128)
    for r in range(n):
        e = row_e[r]
        gu = (A[r] @ _dequant(t, W13q[e], W13s[e], 128, 128).T).astype(np.float32)
        assert np.array_equal(aux["gu"][r], gu), r
        h = (torch.nn.functional.silu(torch.from_numpy(gu[:I]).double()).numpy()
             * gu[I:].astype(np.float64)).astype(np.float32)
        assert np.array_equal(aux["h"][r], h)
        for b in range(I // 128):
            _check_pow2_tile(h[b * 128:(b + 1) * 128], aux["hq"][r, b * 128:(b + 1) * 128],
                             float(aux["hs"][r, b]), t)
        Hd = _dequant(t, aux["hq"][r][None], aux["hs"][r][None], 1, 128)[0]
        yref = torch.from_numpy((_dequant(t, W2q[e], W2s[e], 128, 128) @ Hd).astype(np.float32)) \
            .to(torch.bfloat16).view(torch.uint16).numpy()
        assert np.array_equal(y[r], yref)
    # the FP32-scale mode quantises the same h differently (its scale is amax/448)
    _, aux32 = orc.ffn_fp8(xq, xs, row_e, W13q, W13s, W2q, W2s, want_h=True, pow2=False)
    assert np.array_equal(aux32["gu"], aux["gu"]) and not np.array_equal(aux32["hs"], aux["hs"])

