"""CPU oracle for the DeepSeek-V3-style MoE layer forward (ctypes wrapper over moe_oracle.c).

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's CPU-baseline leg
import this package; the product library and its binding never do, and nothing here
imports the product package.  All arrays are numpy; BF16 data travels as uint16 bit
patterns, E4M3 data as uint8 codes.

Each function names the passage it follows; the C source holds the arithmetic and its
header lists the readings taken where the pages are silent.
"""
import ctypes
import os

import numpy as np

from .build_oracle import build as _build

_lib = None


def lib():
    """Load (building first if needed) the oracle shared library."""
    global _lib
    if _lib is None:
        path = _build()
        L = ctypes.CDLL(path)
        i64, i32, f32, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_float, ctypes.c_void_p
        L.orc_bf16_to_f32.argtypes = [ctypes.c_uint16]
        L.orc_bf16_to_f32.restype = f32
        L.orc_f32_to_bf16.argtypes = [f32]
        L.orc_f32_to_bf16.restype = ctypes.c_uint16
        L.orc_e4m3_to_double.argtypes = [ctypes.c_uint8]
        L.orc_e4m3_to_double.restype = ctypes.c_double
        L.orc_f32_to_e4m3.argtypes = [f32]
        L.orc_f32_to_e4m3.restype = ctypes.c_uint8
        L.orc_num_threads.restype = i32
        L.orc_set_num_threads.argtypes = [i32]
        L.orc_quant_1x128.argtypes = [i64, i64, vp, i32, vp, vp]
        L.orc_quant_1x128_pow2.argtypes = [i64, i64, vp, i32, vp, vp]
        L.orc_quant_128x128.argtypes = [i64, i64, i64, vp, i32, vp, vp]
        L.orc_quant_128x128_pow2.argtypes = [i64, i64, i64, vp, i32, vp, vp]
        L.orc_gate.argtypes = [i64, i32, i32, i32, i32, i32, f32, vp, i32, vp, i32, vp,
                               vp, vp, vp, vp]
        L.orc_permute.argtypes = [i64, i32, i32, i32, vp, vp, vp, vp, vp]
        L.orc_bias_update.argtypes = [i32, i64, i32, vp, vp]
        L.orc_ffn_fp8.argtypes = [i64, i32, i32, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]
        L.orc_ffn_fp8_pow2.argtypes = L.orc_ffn_fp8.argtypes
        L.orc_ffn_f32.argtypes = [i64, i32, i32, vp, vp, vp, vp, vp, vp]
        L.orc_combine.argtypes = [i64, i32, i32, vp, vp, i32, vp, vp]
        L.orc_logfmt_encode.argtypes = [i64, i64, vp, i32, i32, vp, vp, vp, vp]
        L.orc_logfmt_decode.argtypes = [i64, i64, vp, i32, vp, vp, vp]
        _lib = L
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _is_bf16(a):
    if a.dtype == np.uint16:
        return 1
    if a.dtype == np.float32:
        return 0
    raise TypeError("expected float32 or BF16 bits (uint16), got %s" % a.dtype)


def num_threads():
    return lib().orc_num_threads()


def set_num_threads(n):
    lib().orc_set_num_threads(int(n))


# ---------------------------------------------------------------- number formats

def bf16_to_f32(bits):
    """BF16 bit patterns (uint16) -> float32, exact (upper half of the FP32 bits)."""
    bits = _c(bits, np.uint16)
    return (bits.astype(np.uint32) << 16).view(np.float32)


def f32_to_bf16(x):
    """float32 -> BF16 bits, round to nearest even (elementwise through the C routine)."""
    x = _c(x, np.float32)
    L = lib()
    out = np.empty(x.shape, np.uint16)
    flat, of = x.ravel(), out.ravel()
    for i in range(flat.size):
        of[i] = L.orc_f32_to_bf16(float(flat[i]))
    return out


def e4m3_table():
    """The 256 E4M3 code values (OCP OFP8 definition), as float64 (NaN for S.1111.111)."""
    L = lib()
    return np.array([L.orc_e4m3_to_double(c) for c in range(256)], dtype=np.float64)


def f32_to_e4m3(x):
    """float32 -> E4M3 codes, nearest-even with saturation (elementwise C routine)."""
    x = _c(x, np.float32)
    L = lib()
    out = np.empty(x.shape, np.uint8)
    flat, of = x.ravel(), out.ravel()
    for i in range(flat.size):
        of[i] = L.orc_f32_to_e4m3(float(flat[i]))
    return out


# ---------------------------------------------------------------- quantisation

def quant_1x128(x, pow2=False):
    """[Insights into DeepSeek-V3 précis §3.2] 1x128 activation tiles.
    x [rows, cols] float32 or BF16 bits -> (codes uint8 [rows, cols], scales f32 [rows, cols/128]).
    pow2: power-of-two scales (the microscaling form the précis recommends), see moe_oracle.c."""
    x = np.ascontiguousarray(x)
    rows, cols = x.shape
    assert cols % 128 == 0
    q = np.empty((rows, cols), np.uint8)
    s = np.empty((rows, cols // 128), np.float32)
    fn = lib().orc_quant_1x128_pow2 if pow2 else lib().orc_quant_1x128
    fn(rows, cols, _p(x), _is_bf16(x), _p(q), _p(s))
    return q, s


def quant_128x128(w, pow2=False):
    """[Insights into DeepSeek-V3 précis §3.2] 128x128 weight blocks.
    w [n, rows, cols] -> (codes [n, rows, cols], scales f32 [n, rows/128, cols/128]).
    pow2: power-of-two scales, as in quant_1x128."""
    w = np.ascontiguousarray(w)
    if w.ndim == 2:
        w = w[None]
    n, rows, cols = w.shape
    assert rows % 128 == 0 and cols % 128 == 0
    q = np.empty((n, rows, cols), np.uint8)
    s = np.empty((n, rows // 128, cols // 128), np.float32)
    fn = lib().orc_quant_128x128_pow2 if pow2 else lib().orc_quant_128x128
    fn(n, rows, cols, _p(w), _is_bf16(w), _p(q), _p(s))
    return q, s


# ---------------------------------------------------------------- gate, permutation

def gate(x, Wg, bias, n_group, topk_group, top_k, rsf, want_scores=False):
    """[DeepSeek-V3 co-design teardown §2.2, MoEGate] sigmoid gate with the selection-only
    bias and group-limited top-k.  Returns dict(topk_idx [T,K] i32, topk_w [T,K] f32,
    margin [T] f32, scores [T,E] f32 if asked)."""
    x = np.ascontiguousarray(x)
    Wg = np.ascontiguousarray(Wg)
    bias = _c(bias, np.float32)
    T, H = x.shape
    E = Wg.shape[0]
    assert Wg.shape[1] == H and bias.shape == (E,)
    idx = np.empty((T, top_k), np.int32)
    w = np.empty((T, top_k), np.float32)
    margin = np.empty((T,), np.float32)
    scores = np.empty((T, E), np.float32) if want_scores else None
    lib().orc_gate(T, H, E, n_group, topk_group, top_k, float(rsf), _p(x), _is_bf16(x),
                   _p(Wg), _is_bf16(Wg), _p(bias), _p(idx), _p(w), _p(scores), _p(margin))
    out = dict(topk_idx=idx, topk_w=w, margin=margin)
    if want_scores:
        out["scores"] = scores
    return out


def permute(topk_idx, n_experts, has_shared):
    """[DeepSeek-V3 co-design teardown §2.3] counts and expert-major, token-ascending rows.
    Returns dict(counts [E], offs [E+1+has_shared], perm_tok [T*K(+T)], row_of [T,K]).
    Ids outside [0, E) are dropped (row_of -1; the rows they leave at the end of the routed
    part get perm_tok -1), the library's contract for input the gate never produces."""
    topk_idx = _c(topk_idx, np.int32)
    T, K = topk_idx.shape
    E = n_experts
    counts = np.empty((E,), np.int32)
    offs = np.empty((E + 1 + int(bool(has_shared)),), np.int32)
    perm_tok = np.empty((T * K + (T if has_shared else 0),), np.int32)
    row_of = np.empty((T, K), np.int32)
    lib().orc_permute(T, E, K, int(bool(has_shared)), _p(topk_idx), _p(counts), _p(offs),
                      _p(perm_tok), _p(row_of))
    return dict(counts=counts, offs=offs, perm_tok=perm_tok, row_of=row_of)


def bias_update(counts, bias, T, top_k):
    """Load-driven selection-bias update b_i += 1e-3 * sign(mean_load - load_i); returns
    the new bias (the input is not modified)."""
    counts = _c(counts, np.int32)
    b = np.array(bias, dtype=np.float32, copy=True)
    lib().orc_bias_update(counts.shape[0], int(T), int(top_k), _p(counts), _p(b))
    return b


# ---------------------------------------------------------------- experts, combine

def ffn_fp8(aq, as_, row_expert, W13q, W13s, W2q, W2s, want_h=False, pow2=False):
    """[teardown §5.1; précis §3.2] SwiGLU expert rows with blockwise FP8 operands.
    aq [n,H] codes, as_ [n,H/128]; row_expert [n] -> y [n,H] BF16 bits
    (and, if want_h, a dict with gu f32 [n,2I], h f32 [n,I], hq [n,I], hs [n,I/128]).
    pow2: h is re-quantised with power-of-two scales (operands quantised with pow2=True)."""
    aq = _c(aq, np.uint8)
    as_ = _c(as_, np.float32)
    row_expert = _c(row_expert, np.int32)
    W13q, W13s = _c(W13q, np.uint8), _c(W13s, np.float32)
    W2q, W2s = _c(W2q, np.uint8), _c(W2s, np.float32)
    n, H = aq.shape
    I = W2q.shape[2]
    y = np.empty((n, H), np.uint16)
    gu = np.empty((n, 2 * I), np.float32) if want_h else None
    h = np.empty((n, I), np.float32) if want_h else None
    hq = np.empty((n, I), np.uint8) if want_h else None
    hs = np.empty((n, I // 128), np.float32) if want_h else None
    fn = lib().orc_ffn_fp8_pow2 if pow2 else lib().orc_ffn_fp8
    fn(n, H, I, _p(aq), _p(as_), _p(row_expert), _p(W13q), _p(W13s), _p(W2q),
       _p(W2s), _p(gu), _p(h), _p(hq), _p(hs), _p(y))
    if want_h:
        return y, dict(gu=gu, h=h, hq=hq, hs=hs)
    return y


def ffn_f32(x, row_expert, W13, W2, want_h=False):
    """The SwiGLU expert rows with FP32 operands, no quantisation.  x [n,H] f32 -> y [n,H] f32."""
    x = _c(x, np.float32)
    row_expert = _c(row_expert, np.int32)
    W13, W2 = _c(W13, np.float32), _c(W2, np.float32)
    n, H = x.shape
    I = W2.shape[2]
    y = np.empty((n, H), np.float32)
    h = np.empty((n, I), np.float32) if want_h else None
    lib().orc_ffn_f32(n, H, I, _p(x), _p(row_expert), _p(W13), _p(W2), _p(h), _p(y))
    return (y, h) if want_h else y


def combine(yk, w, ysh=None):
    """[teardown §2.3 reverse exchange; précis §3.1 BF16 combine] y = sum_k w_k * y_k + y_shared
    in FP32, slot order.  yk [n,K,H] and ysh [n,H] f32 or BF16 bits; w [n,K].  Returns the
    FP32 sums [n,H] (the caller rounds to BF16 where the layer's output is BF16)."""
    yk = np.ascontiguousarray(yk)
    n, K, H = yk.shape
    isb = _is_bf16(yk)
    if ysh is not None:
        ysh = np.ascontiguousarray(ysh)
        assert ysh.dtype == yk.dtype and ysh.shape == (n, H)
    w = _c(w, np.float32)
    acc = np.empty((n, H), np.float32)
    lib().orc_combine(n, K, H, _p(yk), _p(ysh), isb, _p(w), _p(acc))
    return acc


def round_bf16(x):
    """float32 -> BF16 bits, nearest-even, vectorised form of f32_to_bf16 for large arrays
    (same rule: add 0x7FFF plus the kept LSB, truncate; NaN quieted)."""
    u = _c(x, np.float32).view(np.uint32).astype(np.uint64)
    nan = (u & 0x7FFFFFFF) > 0x7F800000
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
    r[nan] = ((u[nan] >> 16) | 0x40).astype(np.uint16)
    return r


# ---------------------------------------------------------------- whole layer

def quantize_weights(W13, W2, pow2=False):
    """Blockwise-quantise the stacked expert weights once (oracle side)."""
    W13q, W13s = quant_128x128(W13, pow2)
    W2q, W2s = quant_128x128(W2, pow2)
    return W13q, W13s, W2q, W2s


def _take(W, ids):
    """Rows `ids` of a stacked expert tensor: W[ids] for arrays, W(ids) for a callable that
    returns them (lets a caller hand over only the experts a sample touches)."""
    return np.ascontiguousarray(W(ids) if callable(W) else W[ids])


def forward(cfg, x, Wg, bias, W13, W2, sample=None, qweights=None, want_scores=False):
    """The MoE layer forward: gate and permutation over all T tokens, then the expert FFNs
    and the combine for the tokens in `sample` (all tokens when None).  Every output row
    depends only on its own token, so a sample is exact.

    cfg: dict with hidden, inter, n_experts, n_group, topk_group, top_k,
    routed_scaling_factor, has_shared, mode ('fp32' | 'fp8' | 'fp8_pow2': FP8 with
    power-of-two block scales).  x [T,H] (f32 or BF16 bits);
    W13 [E(+1),2I,H], W2 [E(+1),H,I] (the shared expert is the last slot), as arrays or as
    callables ids -> stacked rows.  In fp8 mode `qweights(ids)` may return
    quantize_weights(W13[ids], W2[ids]) from a cache.  Only the experts the sample touches
    are read.  Returns dict with gate outputs, permutation, sample, y (BF16 bits in fp8
    mode, f32 in fp32 mode), yexp [n, K(+1), H] and, in fp8 mode, the sampled xq/xs; with
    want_scores, the gate's scores [T,E] too."""
    g = gate(x, Wg, bias, cfg["n_group"], cfg["topk_group"], cfg["top_k"],
             cfg["routed_scaling_factor"], want_scores=want_scores)
    p = permute(g["topk_idx"], cfg["n_experts"], int(bool(cfg["has_shared"])))
    out = dict(g, **p)
    out.update(experts_and_combine(cfg, x, g, sample, W13, W2, qweights))
    return out


def experts_and_combine(cfg, x, g, sample, W13, W2, qweights=None):
    """The second half of forward(): the expert FFNs (routed slots, then the shared expert)
    and the combine for the tokens in `sample` (all when None), on the routing `g` that
    gate() returned for the whole batch.  Arguments as for forward(); returns dict(sample,
    y, yexp and, in fp8 mode, xq/xs of the sampled tokens and y_f32, the FP32 sums that y
    rounds to BF16)."""
    T = x.shape[0]
    E, K = cfg["n_experts"], cfg["top_k"]
    hs = int(bool(cfg["has_shared"]))
    if sample is None:
        sample = np.arange(T, dtype=np.int64)
    sample = np.asarray(sample, dtype=np.int64)
    n = sample.size
    # one expert row per (sampled token, slot), then the shared expert row
    row_exp = np.empty((n, K + hs), np.int32)
    row_exp[:, :K] = g["topk_idx"][sample]
    if hs:
        row_exp[:, K] = E
    row_exp = row_exp.ravel()
    needed, local = np.unique(row_exp, return_inverse=True)
    local = local.astype(np.int32)
    out = dict(sample=sample)
    if n == 0:
        out.update(y=np.empty((0, x.shape[1]), x.dtype), yexp=None)
        return out
    if cfg["mode"] in ("fp8", "fp8_pow2"):
        pow2 = cfg["mode"] == "fp8_pow2"
        xq, xs = quant_1x128(np.ascontiguousarray(x[sample]), pow2)
        if qweights is not None:
            qw = qweights(needed)
        else:
            qw = quantize_weights(_take(W13, needed), _take(W2, needed), pow2)
        rep = np.repeat(np.arange(n), K + hs)
        yrows = ffn_fp8(xq[rep], xs[rep], local, *qw, pow2=pow2).reshape(n, K + hs, -1)
        acc = combine(yrows[:, :K], g["topk_w"][sample],
                      np.ascontiguousarray(yrows[:, K]) if hs else None)
        out.update(y=round_bf16(acc), y_f32=acc, yexp=yrows, xq=xq, xs=xs)
    else:
        xr = np.ascontiguousarray(np.repeat(x[sample], K + hs, axis=0))
        yrows = ffn_f32(xr, local, _take(W13, needed), _take(W2, needed)).reshape(n, K + hs, -1)
        acc = combine(yrows[:, :K], g["topk_w"][sample],
                      np.ascontiguousarray(yrows[:, K]) if hs else None)
        out.update(y=acc, yexp=yrows)
    return out


# ---------------------------------------------------------------- LogFMT codec

def logfmt_encode(x, n_bits):
    """[Insights into DeepSeek-V3 précis §3.2, LogFMT-nBit] per 1x128 tile: min and max of the
    natural log of the non-zero magnitudes (min held above max - ln 2^32), Step = (max - min) /
    (2^(n-1) - 2), each value coded with the K whose exp(min + Step (K-1)) is nearest in linear
    space (K = 0: zero), sign in the top bit.  x [rows, cols] float32 or BF16 bits.
    Returns dict(codes uint16 [rows, cols], lmin f32 [rows, cols/128], step f32 [...],
    margin f32 [rows, cols]: distance to the decision midpoint as a fraction of the gap)."""
    x = np.ascontiguousarray(x)
    rows, cols = x.shape
    assert cols % 128 == 0 and 3 <= n_bits <= 16
    codes = np.empty((rows, cols), np.uint16)
    lmin = np.empty((rows, cols // 128), np.float32)
    step = np.empty((rows, cols // 128), np.float32)
    margin = np.empty((rows, cols), np.float32)
    lib().orc_logfmt_encode(rows, cols, _p(x), _is_bf16(x), int(n_bits), _p(codes), _p(lmin), _p(step),
                            _p(margin))
    return dict(codes=codes, lmin=lmin, step=step, margin=margin)


def logfmt_decode(codes, lmin, step, n_bits):
    """Inverse of logfmt_encode: +-exp(min + Step (K-1)) (0 for K = 0), float32 [rows, cols]."""
    codes = _c(codes, np.uint16)
    rows, cols = codes.shape
    out = np.empty((rows, cols), np.float32)
    lib().orc_logfmt_decode(rows, cols, _p(codes), int(n_bits), _p(_c(lmin, np.float32)),
                            _p(_c(step, np.float32)), _p(out))
    return out
