"""Comparison helpers for the GPU-vs-oracle parity tests.

Tolerances (written here, used by every parity test):
  - routing indices, per-expert counts, permutation order, quantised codes of the same
    FP32 inputs and the bias update: bit-exact, except on tokens whose selection margin in
    the oracle (k-th vs (k+1)-th selection score, or topk_group-th vs next group score) is
    below ROUTING_MARGIN -- there the GPU's choice must still be a valid one;
  - routing weights: |gpu - ref| <= WEIGHT_ATOL * routed_scaling_factor (FP32 logits summed in
    another order than the oracle's double sum);
  - layer and expert outputs: max|gpu - ref| / max|ref| <= 5e-3 (FP8 path) or 1e-3 (FP32).
"""
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


def check_permutation(p_gpu, idx, orc, n_experts, has_shared):
    """GPU permutation vs the oracle's permutation of the SAME routing: bit-exact."""
    ref = orc.permute(idx, n_experts, has_shared)
    for k in ("offs", "perm_tok"):
        assert np.array_equal(p_gpu[k], ref[k]), k
    assert np.array_equal(p_gpu["row_of"].reshape(ref["row_of"].shape), ref["row_of"])
    return ref
