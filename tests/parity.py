"""Comparison helpers for the GPU-vs-oracle parity tests.

Tolerances (written here, used by every parity test):
  - routing indices, per-expert counts, permutation order, quantised codes of the same
    FP32 inputs and the bias update: bit-exact, except on tokens whose selection margin in
    the oracle (k-th vs (k+1)-th selection score, or topk_group-th vs next group score) is
    below ROUTING_MARGIN -- there the GPU's choice must still be a valid one
    (check_flagged_routing: a top choice within the margin, with matching weights);
  - routing weights: |gpu - ref| <= WEIGHT_ATOL * routed_scaling_factor (FP32 logits summed in
    another order than the oracle's double sum);
  - layer and expert outputs: max|gpu - ref| / max|ref| <= 5e-3 (FP8 path) or 1e-3 (FP32);
    for the BF16 layer output, ref is the oracle's FP32 sum before its own BF16 rounding:
    comparing two independently rounded BF16 values would charge up to one BF16 unit in the
    last place (0.4-0.8 % of an element) of pure output-format rounding against a 0.5 % bar.
"""
import itertools

import numpy as np
import torch

ROUTING_MARGIN = 1e-5
WEIGHT_ATOL = 2e-5
TOL_FP8 = 5e-3
TOL_FP32 = 1e-3


def to_host(t):
    """Device tensor -> numpy (BF16 as uint16 bits)."""
    t = t.detach()
    if t.dtype == torch.bfloat16:
        t = t.view(torch.uint16)
    return t.cpu().numpy()


def bf16_bits_to_f32(a):
    return (np.asarray(a, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def rel_err(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    den = np.max(np.abs(ref))
    if den == 0:
        return float(np.max(np.abs(got)))
    return float(np.max(np.abs(got - ref)) / den)


def check_routing(g_idx, g_w, ref, rsf):
    """Compare the GPU's routing with the oracle's.  Returns the mask of flagged tokens (margin
    below ROUTING_MARGIN).  On unflagged tokens the sets of chosen experts must agree and the
    weight paired with each expert must agree within WEIGHT_ATOL * rsf."""
    flagged = ref["margin"] < ROUTING_MARGIN
    gi = np.sort(g_idx, axis=1)
    ri = np.sort(ref["topk_idx"], axis=1)
    bad = np.nonzero(np.any(gi != ri, axis=1) & ~flagged)[0]
    assert bad.size == 0, "routing differs on %d unflagged tokens, e.g. %s: gpu %s ref %s" % (
        bad.size, bad[:3], g_idx[bad[:1]], ref["topk_idx"][bad[:1]])
    ok = ~flagged
    gw = np.take_along_axis(g_w, np.argsort(g_idx, axis=1), 1)
    rw = np.take_along_axis(ref["topk_w"], np.argsort(ref["topk_idx"], axis=1), 1)
    err = np.max(np.abs(gw[ok] - rw[ok])) if ok.any() else 0.0
    assert err <= WEIGHT_ATOL * rsf, "routing weights differ by %g" % err
    return flagged


def check_valid_routing(g_idx, n_experts, n_group, topk_group):
    """Every token's experts are distinct, in range, and lie in at most topk_group groups."""
    assert np.all((g_idx >= 0) & (g_idx < n_experts))
    s = np.sort(g_idx, axis=1)
    assert np.all(s[:, 1:] != s[:, :-1]) if g_idx.shape[1] > 1 else True
    groups = g_idx // (n_experts // n_group)
    for row in groups:
        assert len(set(row.tolist())) <= topk_group


def _top2_group_scores(c, n_group):
    """Group score of [DeepSeek-V3 co-design teardown §2.2]: the sum of the two largest
    selection scores of each group (float32, larger first)."""
    g = np.sort(c.reshape(n_group, -1), axis=1)[:, ::-1]
    return (g[:, 0] + g[:, 1]).astype(np.float32)


def check_flagged_routing(g_idx, g_w, ref, bias, n_group, topk_group, rsf, tol=ROUTING_MARGIN):
    """On the tokens the oracle flags (selection margin below tol), where several choices are
    correct up to the rounding of the scores, the GPU's choice must be one of them.  With the
    oracle's scores s (ref["scores"]) and selection scores c = s + bias:
      - the GPU's experts lie in a set S of topk_group groups that is a top-topk_group choice
        by group score within tol (every group of S at least the cut - tol, every other group
        at most the lowest of S + tol);
      - their summed selection score is within top_k * tol of the best top_k sum inside S;
      - the weight paired with each chosen expert is its score normalised over the chosen set
        (top_k > 1) times rsf, within WEIGHT_ATOL * rsf.
    Returns the number of tokens checked."""
    flagged = np.nonzero(ref["margin"] < tol)[0]
    if flagged.size == 0:
        return 0
    assert "scores" in ref, "the oracle's scores are needed to validate flagged tokens"
    T, K = g_idx.shape
    E = ref["scores"].shape[1]
    gsz = E // n_group
    for t in flagged:
        s = ref["scores"][t].astype(np.float32)
        c = (s + bias).astype(np.float32)
        gs = _top2_group_scores(c, n_group)
        cut = np.sort(gs)[::-1][topk_group - 1]
        used = set((g_idx[t] // gsz).tolist())
        ok = False
        for S in itertools.combinations(range(n_group), topk_group):
            if not used <= set(S):
                continue
            lo = min(gs[g] for g in S)
            if lo < cut - tol or any(gs[g] > lo + tol for g in range(n_group) if g not in S):
                continue
            allowed = np.array([e for e in range(E) if e // gsz in S])
            best = np.sort(c[allowed].astype(np.float64))[::-1][:K].sum()
            if c[g_idx[t]].astype(np.float64).sum() >= best - K * tol:
                ok = True
                break
        assert ok, "token %d: the GPU's experts %s are not a valid choice" % (t, g_idx[t].tolist())
        sel = s[g_idx[t]].astype(np.float64)
        want = sel / (sel.sum() + 1e-20) * rsf if K > 1 else sel * rsf
        err = np.max(np.abs(g_w[t] - want))
        assert err <= WEIGHT_ATOL * rsf, "token %d: weights differ by %g" % (t, err)
    return int(flagged.size)


def check_permutation(p_gpu, idx, orc, n_experts, has_shared):
    """GPU permutation vs the oracle's permutation of the SAME routing: bit-exact."""
    ref = orc.permute(idx, n_experts, has_shared)
    for k in ("offs", "perm_tok"):
        assert np.array_equal(p_gpu[k], ref[k]), k
    assert np.array_equal(p_gpu["row_of"].reshape(ref["row_of"].shape), ref["row_of"])
    return ref
