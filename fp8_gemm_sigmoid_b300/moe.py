"""Python binding of libmoe (ctypes): argument marshalling only.

Every function here has the name of the C entry point it calls (include/moe.h), takes
torch tensors that already live on the GPU, passes their device pointers and the current
torch stream, and raises MoEError on a non-OK status.  All arithmetic runs in libmoe's
CUDA kernels; if the library is missing this module raises instead of computing anything
another way.
"""
import contextlib
import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe.so")
CHECKS_LIB_PATH = os.path.join(_HERE, "libmoe_checks.so")  # the -DMOE_CHECKS debug build

MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_WORKSPACE, MOE_ERR_CUDA, MOE_ERR_TIMEOUT = range(6)
MOE_FP32, MOE_FP8_BLOCK, MOE_MXFP8 = 0, 1, 2
MOE_EPI_SWIGLU_QUANT, MOE_EPI_STORE = 0, 1
MOE_GATE_QUANT_MIN_TOKENS = 6144  # moe_forward fuses the quantisation into the gate from here up


class MoEError(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        super().__init__("%s failed: %s" % (fn, _lib_handle().moe_status_string(status).decode()))


class moe_config(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int32), ("inter", ctypes.c_int32),
                ("n_experts", ctypes.c_int32), ("n_group", ctypes.c_int32),
                ("topk_group", ctypes.c_int32), ("top_k", ctypes.c_int32),
                ("routed_scaling_factor", ctypes.c_float), ("has_shared", ctypes.c_int32),
                ("mode", ctypes.c_int32)]


class moe_weights(ctypes.Structure):
    _fields_ = [("Wg", ctypes.c_void_p), ("W13", ctypes.c_void_p), ("W13_s", ctypes.c_void_p),
                ("W2", ctypes.c_void_p), ("W2_s", ctypes.c_void_p)]


_L = None
_vp, _i64, _i32, _sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_size_t
_cfgp = ctypes.POINTER(moe_config)

_SIGS = {
    "moe_config_validate": [_cfgp],
    "moe_workspace_size": [_cfgp, _i64, ctypes.POINTER(_sz)],
    "moe_gate": [_cfgp, _i64, _vp, _vp, _vp, _vp, _vp, _vp, _vp],
    "moe_gate_quant": [_cfgp, _i64, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp],
    "moe_quant_1x128": [_i64, _i64, _vp, _vp, _vp, _vp],
    "moe_quant_128x128": [_i64, _i64, _i64, _vp, _vp, _vp, _vp],
    "moe_quant_1x128_pow2": [_i64, _i64, _vp, _vp, _vp, _vp],
    "moe_quant_128x128_pow2": [_i64, _i64, _i64, _vp, _vp, _vp, _vp],
    "moe_grouped_gemm_mxfp8": [_i32, _vp, _i64, _i32, _i32, _vp, _vp, _vp, _vp, _i32, _vp, _vp, _vp],
    "moe_grouped_gemm_fp8_gather": [_i32, _vp, _i64, _i32, _i32, _vp, _i64, _vp, _vp, _vp, _vp, _i32, _vp, _vp,
                                    _vp],
    "moe_grouped_gemm_mxfp8_gather": [_i32, _vp, _i64, _i32, _i32, _vp, _i64, _vp, _vp, _vp, _vp, _i32, _vp,
                                      _vp, _vp],
    "moe_permute": [_cfgp, _i64, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp],
    "moe_grouped_gemm_fp8": [_i32, _vp, _i64, _i32, _i32, _vp, _vp, _vp, _vp, _i32, _vp, _vp,
                             _vp, _sz, _vp],
    "moe_grouped_gemm_f32": [_i32, _vp, _i64, _i32, _i32, _vp, _vp, _i32, _vp, _vp, _sz, _vp],
    "moe_combine": [_cfgp, _i64, _vp, _vp, _vp, _vp, _vp, _vp],
    "moe_bias_update": [_cfgp, _i64, _vp, _vp, _vp],
    "moe_forward": [_cfgp, _i64, _vp, ctypes.POINTER(moe_weights), _vp, _i32, _vp, _vp, _vp,
                    _vp, _vp, _sz, _vp],
    "moe_device_error": [ctypes.POINTER(_i32)],
    "moe_selftest_wait_timeout": [_i64, _vp],
    "moe_pipeline_workspace_size": [_cfgp, _i64, ctypes.POINTER(_sz)],
    "moe_pipeline_create": [_cfgp, _i64, _vp, _sz, _vp, ctypes.POINTER(_vp)],
    "moe_pipeline_submit": [_vp, _i64, _vp, ctypes.POINTER(moe_weights), _vp, _i32, _vp, _vp, _vp, _vp],
    "moe_pipeline_wait": [_vp],
    "moe_pipeline_destroy": [_vp],
    "moe_gather_rows": [_i64, _i64, _vp, _vp, _vp, _vp],
    "moe_logfmt_encode": [_i32, _i64, _i64, _vp, _vp, _vp, _vp, _vp],
    "moe_logfmt_decode": [_i32, _i64, _i64, _vp, _vp, _vp, _vp, _vp],
}


def _load(path):
    if not os.path.exists(path):
        raise RuntimeError("%s is not built; run `python -m fp8_gemm_sigmoid_b300.build%s`"
                           % (path, " --checks" if path == CHECKS_LIB_PATH else ""))
    L = ctypes.CDLL(path)
    L.moe_status_string.argtypes = [ctypes.c_int]
    L.moe_status_string.restype = ctypes.c_char_p
    for name, args in _SIGS.items():
        f = getattr(L, name)
        f.argtypes = args
        f.restype = ctypes.c_int
    return L


def _lib_handle():
    global _L
    if _L is None:
        _L = _load(LIB_PATH)
    return _L


_CHECKS = None


@contextlib.contextmanager
def checks_library():
    """Routes this module's calls to libmoe_checks.so (the same kernels with the MOE_CHECKS
    index checks compiled in) inside the with-block, then back to libmoe.so.  Both libraries
    stay loaded side by side; each has its own device error words."""
    global _L, _CHECKS
    if _CHECKS is None:
        _CHECKS = _load(CHECKS_LIB_PATH)
    prev = _lib_handle()
    _L = _CHECKS
    try:
        yield _CHECKS
    finally:
        _L = prev


def exported_symbols():
    """Names of the ABI entry points this binding expects libmoe.so to export."""
    return ["moe_status_string"] + list(_SIGS)


def _check(name, status):
    if status != MOE_OK:
        raise MoEError(name, status)


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("libmoe takes device tensors; got a %s tensor" % t.device)
    if not t.is_contiguous():
        raise ValueError("libmoe takes contiguous tensors")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def make_config(cfg):
    """moe_config from a workload dict (hidden, inter, n_experts, n_group, topk_group,
    top_k, routed_scaling_factor, has_shared, mode 'fp32' | 'fp8' | 'mxfp8')."""
    mode = {"fp32": MOE_FP32, "fp8": MOE_FP8_BLOCK, "mxfp8": MOE_MXFP8}[cfg["mode"]]
    return moe_config(cfg["hidden"], cfg["inter"], cfg["n_experts"], cfg["n_group"],
                      cfg["topk_group"], cfg["top_k"], float(cfg["routed_scaling_factor"]),
                      int(cfg["has_shared"]), mode)


def _cfg(c):
    return c if isinstance(c, moe_config) else make_config(c)


def moe_config_validate(cfg):
    return _lib_handle().moe_config_validate(ctypes.byref(_cfg(cfg))) == MOE_OK


def moe_workspace_size(cfg, T):
    n = _sz(0)
    _check("moe_workspace_size", _lib_handle().moe_workspace_size(ctypes.byref(_cfg(cfg)), int(T), ctypes.byref(n)))
    return n.value


def moe_gate(cfg, x, Wg, bias, topk_idx, topk_w, counts, stream=None):
    T = x.shape[0]
    _check("moe_gate", _lib_handle().moe_gate(ctypes.byref(_cfg(cfg)), T, _ptr(x), _ptr(Wg), _ptr(bias),
                                              _ptr(topk_idx), _ptr(topk_w), _ptr(counts), _stream(stream)))


def moe_gate_quant(cfg, x, Wg, bias, topk_idx, topk_w, counts, xq, xs, stream=None):
    """moe_gate plus the 1x128 quantisation of x (xq [T, H] codes, xs [T, H/128] scales) in one
    pass over x; raises MoEError with status MOE_ERR_UNSUPPORTED outside the fused kernel."""
    T = x.shape[0]
    _check("moe_gate_quant", _lib_handle().moe_gate_quant(
        ctypes.byref(_cfg(cfg)), T, _ptr(x), _ptr(Wg), _ptr(bias), _ptr(topk_idx), _ptr(topk_w),
        _ptr(counts), _ptr(xq), _ptr(xs), _stream(stream)))


def moe_quant_1x128(x, q, s, stream=None):
    rows, cols = x.shape
    _check("moe_quant_1x128", _lib_handle().moe_quant_1x128(rows, cols, _ptr(x), _ptr(q), _ptr(s), _stream(stream)))


def moe_quant_128x128(w, q, s, stream=None, pow2=False):
    n, rows, cols = w.shape if w.dim() == 3 else (1, *w.shape)
    name = "moe_quant_128x128_pow2" if pow2 else "moe_quant_128x128"
    _check(name, getattr(_lib_handle(), name)(n, rows, cols, _ptr(w), _ptr(q), _ptr(s), _stream(stream)))


def moe_quant_1x128_pow2(x, q, s, stream=None):
    rows, cols = x.shape
    _check("moe_quant_1x128_pow2", _lib_handle().moe_quant_1x128_pow2(rows, cols, _ptr(x), _ptr(q), _ptr(s),
                                                                      _stream(stream)))


def moe_grouped_gemm_mxfp8(n_groups, offs, rows, N, Kdim, A, As, W, Ws, epilogue, out, out_s, stream=None):
    _check("moe_grouped_gemm_mxfp8", _lib_handle().moe_grouped_gemm_mxfp8(
        int(n_groups), _ptr(offs), int(rows), int(N), int(Kdim), _ptr(A), _ptr(As), _ptr(W), _ptr(Ws),
        int(epilogue), _ptr(out), _ptr(out_s), _stream(stream)))


def moe_permute(cfg, T, topk_idx, counts, xq, xs, offs, perm_tok, row_of, aq, as_, ws, stream=None):
    _check("moe_permute", _lib_handle().moe_permute(
        ctypes.byref(_cfg(cfg)), int(T), _ptr(topk_idx), _ptr(counts), _ptr(xq), _ptr(xs), _ptr(offs),
        _ptr(perm_tok), _ptr(row_of), _ptr(aq), _ptr(as_), _ptr(ws), ws.numel() * ws.element_size(),
        _stream(stream)))


def moe_grouped_gemm_fp8(n_groups, offs, rows, N, Kdim, A, As, W, Ws, epilogue, out, out_s, ws,
                         stream=None):
    _check("moe_grouped_gemm_fp8", _lib_handle().moe_grouped_gemm_fp8(
        int(n_groups), _ptr(offs), int(rows), int(N), int(Kdim), _ptr(A), _ptr(As), _ptr(W), _ptr(Ws),
        int(epilogue), _ptr(out), _ptr(out_s), _ptr(ws),
        0 if ws is None else ws.numel() * ws.element_size(), _stream(stream)))


def moe_grouped_gemm_fp8_gather(n_groups, offs, rows, N, Kdim, perm_tok, X, Xs, W, Ws, epilogue, out, out_s,
                                stream=None, mx=False):
    """Row r of A is X[perm_tok[r]] (X [T, Kdim] codes, Xs [T, Kdim/128] row-major scales);
    mx: the power-of-two (MXFP8) kernel."""
    name = "moe_grouped_gemm_mxfp8_gather" if mx else "moe_grouped_gemm_fp8_gather"
    _check(name, getattr(_lib_handle(), name)(
        int(n_groups), _ptr(offs), int(rows), int(N), int(Kdim), _ptr(perm_tok), int(X.shape[0]), _ptr(X),
        _ptr(Xs), _ptr(W), _ptr(Ws), int(epilogue), _ptr(out), _ptr(out_s), _stream(stream)))


def moe_grouped_gemm_f32(n_groups, offs, rows, N, Kdim, A, W, epilogue, out, ws, stream=None):
    _check("moe_grouped_gemm_f32", _lib_handle().moe_grouped_gemm_f32(
        int(n_groups), _ptr(offs), int(rows), int(N), int(Kdim), _ptr(A), _ptr(W), int(epilogue),
        _ptr(out), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))


def moe_combine(cfg, T, yexp, row_of, topk_w, yshared, y, stream=None):
    """yexp: the routed expert rows [T*K, H] (extra rows after them are ignored); yshared: the
    shared expert's rows [T, H] (None without a shared expert)."""
    _check("moe_combine", _lib_handle().moe_combine(ctypes.byref(_cfg(cfg)), int(T), _ptr(yexp), _ptr(row_of),
                                                    _ptr(topk_w), _ptr(yshared), _ptr(y), _stream(stream)))


def moe_bias_update(cfg, T, counts, bias, stream=None):
    _check("moe_bias_update", _lib_handle().moe_bias_update(ctypes.byref(_cfg(cfg)), int(T), _ptr(counts),
                                                            _ptr(bias), _stream(stream)))


def moe_forward(cfg, x, weights, bias, update_bias, y, topk_idx, topk_w, counts, ws, stream=None):
    """weights: dict with Wg, W13, W2 and (FP8) W13_s, W2_s device tensors."""
    w = moe_weights(_ptr(weights["Wg"]), _ptr(weights["W13"]), _ptr(weights.get("W13_s")),
                    _ptr(weights["W2"]), _ptr(weights.get("W2_s")))
    _check("moe_forward", _lib_handle().moe_forward(
        ctypes.byref(_cfg(cfg)), x.shape[0], _ptr(x), ctypes.byref(w), _ptr(bias), int(bool(update_bias)),
        _ptr(y), _ptr(topk_idx), _ptr(topk_w), _ptr(counts), _ptr(ws), ws.numel() * ws.element_size(),
        _stream(stream)))


def moe_permute_noalloc(cfg, T, topk_idx, xq, xs, offs, perm_tok, row_of, aq, as_, stream=None):
    """moe_permute without a workspace: its counters live in libmoe's fixed device array
    (see include/moe.h for the size limit and the rule that overlapping calls race)."""
    f = _lib_handle().moe_permute_noalloc
    f.argtypes = [_cfgp, _i64, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp]
    f.restype = ctypes.c_int
    _check("moe_permute_noalloc", f(ctypes.byref(_cfg(cfg)), int(T), _ptr(topk_idx), _ptr(xq), _ptr(xs),
                                    _ptr(offs), _ptr(perm_tok), _ptr(row_of), _ptr(aq), _ptr(as_),
                                    _stream(stream)))


def moe_gather_rows(idx, src, dst, stream=None):
    """dst[r] = src[idx[r]] row by row (zero rows where idx < 0); src, dst 2-D."""
    row_bytes = src.shape[1] * src.element_size()
    _check("moe_gather_rows", _lib_handle().moe_gather_rows(int(idx.numel()), int(row_bytes), _ptr(idx),
                                                            _ptr(src), _ptr(dst), _stream(stream)))


def moe_logfmt_encode(n_bits, x, codes, lmin, step, stream=None):
    """x [rows, cols] BF16 (bits as uint16); codes uint8 (n_bits <= 8) or uint16 [rows, cols];
    lmin, step float32 [rows, cols/128]."""
    rows, cols = x.shape
    _check("moe_logfmt_encode", _lib_handle().moe_logfmt_encode(
        int(n_bits), rows, cols, _ptr(x), _ptr(codes), _ptr(lmin), _ptr(step), _stream(stream)))


def moe_logfmt_decode(n_bits, codes, lmin, step, y, stream=None):
    rows, cols = codes.shape
    _check("moe_logfmt_decode", _lib_handle().moe_logfmt_decode(
        int(n_bits), rows, cols, _ptr(codes), _ptr(lmin), _ptr(step), _ptr(y), _stream(stream)))


def moe_device_error():
    code = _i32(0)
    _check("moe_device_error", _lib_handle().moe_device_error(ctypes.byref(code)))
    return code.value


# ---------------------------------------------------------------- allocation helpers
# (plain torch allocations of the buffers the entry points write; no arithmetic)

def empty_outputs(cfg, T, device="cuda"):
    K, E, H = cfg["top_k"], cfg["n_experts"], cfg["hidden"]
    dt = torch.float32 if cfg["mode"] == "fp32" else torch.bfloat16
    return dict(y=torch.empty((T, H), dtype=dt, device=device),
                topk_idx=torch.empty((T, K), dtype=torch.int32, device=device),
                topk_w=torch.empty((T, K), dtype=torch.float32, device=device),
                counts=torch.empty((E,), dtype=torch.int32, device=device))


def workspace(cfg, T, device="cuda"):
    return torch.empty((moe_workspace_size(cfg, T),), dtype=torch.uint8, device=device)


def quantize_weights(W13, W2, stream=None, pow2=False):
    """FP8 copies of the stacked BF16 expert weights via moe_quant_128x128 (moe_quant_128x128_pow2
    with pow2: the power-of-two scales of the MXFP8 mode)."""
    out = {}
    for name, W in (("W13", W13), ("W2", W2)):
        n, R, C = W.shape
        q = torch.empty((n, R, C), dtype=torch.uint8, device=W.device)
        s = torch.empty((n, R // 128, C // 128), dtype=torch.float32, device=W.device)
        moe_quant_128x128(W.view(torch.uint16) if W.dtype == torch.bfloat16 else W, q, s, stream, pow2=pow2)
        out[name], out[name + "_s"] = q, s
    return out


# ---------------------------------------------------------------- host-buffer pipeline

def _host_ptr(t):
    if t is None:
        return None
    if t.is_cuda:
        raise ValueError("moe_pipeline_submit takes host tensors; got a %s tensor" % t.device)
    if not t.is_contiguous():
        raise ValueError("libmoe takes contiguous tensors")
    return ctypes.c_void_p(t.data_ptr())


def moe_pipeline_workspace_size(cfg, max_T):
    n = _sz(0)
    _check("moe_pipeline_workspace_size", _lib_handle().moe_pipeline_workspace_size(
        ctypes.byref(_cfg(cfg)), int(max_T), ctypes.byref(n)))
    return n.value


class MoEPipeline:
    """moe_pipeline_create / submit / wait / destroy: the layer from and to (pinned) host
    tensors, with consecutive batches' copies overlapping each other's compute."""

    def __init__(self, cfg, max_T, ws=None, stream=None, device="cuda"):
        self.cfg = _cfg(cfg)
        self.ws = ws if ws is not None else torch.empty(
            (moe_pipeline_workspace_size(cfg, max_T),), dtype=torch.uint8, device=device)
        self.handle = _vp(0)
        _check("moe_pipeline_create", _lib_handle().moe_pipeline_create(
            ctypes.byref(self.cfg), int(max_T), _ptr(self.ws), self.ws.numel() * self.ws.element_size(),
            _stream(stream), ctypes.byref(self.handle)))
        self._keep = []

    def submit(self, x_host, weights, bias, update_bias, y_host, topk_idx_host, topk_w_host, counts_host):
        w = moe_weights(_ptr(weights["Wg"]), _ptr(weights["W13"]), _ptr(weights.get("W13_s")),
                        _ptr(weights["W2"]), _ptr(weights.get("W2_s")))
        self._keep = [w]
        _check("moe_pipeline_submit", _lib_handle().moe_pipeline_submit(
            self.handle, int(x_host.shape[0]), _host_ptr(x_host), ctypes.byref(w), _ptr(bias),
            int(update_bias), _host_ptr(y_host), _host_ptr(topk_idx_host), _host_ptr(topk_w_host),
            _host_ptr(counts_host)))

    def wait(self):
        _check("moe_pipeline_wait", _lib_handle().moe_pipeline_wait(self.handle))

    def close(self):
        if self.handle:
            _check("moe_pipeline_destroy", _lib_handle().moe_pipeline_destroy(self.handle))
            self.handle = _vp(0)

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def moe_selftest_wait_timeout(budget_cycles, stream=None):
    _check("moe_selftest_wait_timeout", _lib_handle().moe_selftest_wait_timeout(int(budget_cycles), _stream(stream)))
