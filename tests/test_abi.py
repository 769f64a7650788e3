"""The C-ABI library: it builds, loads and exports every entry point include/moe.h declares,
and its host-side argument checks reject bad input without touching a GPU."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def moe():
    from fp8_gemm_sigmoid_b300 import build, moe as m
    build.build()
    return m


def header_symbols():
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    return sorted(set(re.findall(r"MOE_API\s+[\w\s\*]+?\b(moe_\w+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = header_symbols()
    for n in ("moe_gate", "moe_quant_1x128", "moe_quant_128x128", "moe_permute",
              "moe_grouped_gemm_fp8", "moe_combine", "moe_bias_update", "moe_forward",
              "moe_workspace_size", "moe_status_string"):
        assert n in names, n


def test_library_exports_every_header_symbol(moe):
    lib = ctypes.CDLL(moe.LIB_PATH)
    for n in header_symbols():
        assert hasattr(lib, n), n
    out = subprocess.run(["nm", "-D", "--defined-only", moe.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\sT\s(moe_\w+)", out))
    assert set(header_symbols()) <= exported
    assert set(moe.exported_symbols()) <= exported


def test_config_validation(moe):
    from fp8_gemm_sigmoid_b300 import synthetic as sy
    for name in sy.CONFIGS:
        assert moe.moe_config_validate(sy.config(name))
    base = sy.config("v3_prefill")
    bad = [dict(base, n_group=7), dict(base, topk_group=9), dict(base, top_k=129),
           dict(base, hidden=7000), dict(base, inter=100), dict(base, n_experts=8, n_group=8),
           dict(base, has_shared=2), dict(base, top_k=0), dict(base, n_experts=2048, n_group=32)]
    for c in bad:
        assert not moe.moe_config_validate(c), c


def test_workspace_size_grows_with_tokens(moe):
    from fp8_gemm_sigmoid_b300 import synthetic as sy
    c = sy.config("v3_prefill")
    a, b = moe.moe_workspace_size(c, 128), moe.moe_workspace_size(c, 16384)
    assert 0 < a < b
    # at least the permuted FP8 rows, their BF16 outputs and the FFN activations
    R = 16384 * 9
    assert b >= R * (7168 + 2 * 7168 + 2048)


def test_host_side_argument_checks(moe):
    L = moe._lib_handle()
    vp = ctypes.c_void_p
    # shapes that break the 1x128 / 128x128 contract are rejected before any launch
    assert L.moe_quant_1x128(4, 100, vp(16), vp(16), vp(16), None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_quant_1x128(4, 128, None, vp(16), vp(16), None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_quant_1x128(4, 128, vp(17), vp(16), vp(16), None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_quant_128x128(1, 100, 128, vp(16), vp(16), vp(16), None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_grouped_gemm_fp8(0, vp(16), 10, 256, 256, vp(16), vp(16), vp(16), vp(16), 0,
                                  vp(16), vp(16), vp(16), 1 << 20, None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_grouped_gemm_fp8(2, vp(16), 10, 256, 256, vp(16), vp(16), vp(16), vp(16), 7,
                                  vp(16), vp(16), vp(16), 1 << 20, None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_grouped_gemm_fp8(2, vp(16), 10, 256, 200, vp(16), vp(16), vp(16), vp(16), 0,
                                  vp(16), vp(16), vp(16), 0, None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_grouped_gemm_fp8(2, vp(16), 10, 256, 256, vp(16), vp(16), vp(16), vp(16), 0,
                                  vp(16), vp(17), vp(16), 0, None) == moe.MOE_ERR_INVALID_ARG
    # more groups than the in-kernel tile schedule holds
    assert L.moe_grouped_gemm_fp8(1041, vp(16), 10, 256, 256, vp(16), vp(16), vp(16), vp(16), 0,
                                  vp(16), vp(16), vp(16), 0, None) == moe.MOE_ERR_UNSUPPORTED
    from fp8_gemm_sigmoid_b300 import synthetic as sy
    cfg = moe.make_config(sy.config("v3_prefill"))
    need = ctypes.c_size_t(0)
    assert L.moe_workspace_size(ctypes.byref(cfg), 1000, ctypes.byref(need)) == moe.MOE_OK
    assert L.moe_permute(ctypes.byref(cfg), 1000, vp(16), vp(16), vp(16), vp(16), vp(16), vp(16),
                         vp(16), vp(16), vp(16), vp(16), need.value - 1, None) == moe.MOE_ERR_WORKSPACE
    assert L.moe_workspace_size(ctypes.byref(cfg), -1, ctypes.byref(need)) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_status_string(moe.MOE_ERR_TIMEOUT).startswith(b"MOE_ERR_TIMEOUT")


def test_pipeline_host_side_checks(moe):
    L = moe._lib_handle()
    from fp8_gemm_sigmoid_b300 import synthetic as sy
    cfg = moe.make_config(sy.config("v3_prefill"))
    a, b = ctypes.c_size_t(0), ctypes.c_size_t(0)
    assert L.moe_pipeline_workspace_size(ctypes.byref(cfg), 1000, ctypes.byref(a)) == moe.MOE_OK
    assert L.moe_pipeline_workspace_size(ctypes.byref(cfg), 2000, ctypes.byref(b)) == moe.MOE_OK
    layer = ctypes.c_size_t(0)
    assert L.moe_workspace_size(ctypes.byref(cfg), 1000, ctypes.byref(layer)) == moe.MOE_OK
    # the layer workspace plus two slots of x and y (BF16 [T, H]) at least
    assert a.value >= layer.value + 4 * 1000 * 7168 * 2 and b.value > a.value
    assert L.moe_pipeline_workspace_size(ctypes.byref(cfg), 0, ctypes.byref(a)) == moe.MOE_ERR_INVALID_ARG
    h = ctypes.c_void_p(0)
    # rejected before any CUDA call: no workspace, a misaligned one, one too small
    assert L.moe_pipeline_create(ctypes.byref(cfg), 1000, None, b.value, None, ctypes.byref(h)) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_pipeline_create(ctypes.byref(cfg), 1000, ctypes.c_void_p(17), b.value, None,
                                 ctypes.byref(h)) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_pipeline_create(ctypes.byref(cfg), 1000, ctypes.c_void_p(16), 100, None,
                                 ctypes.byref(h)) == moe.MOE_ERR_WORKSPACE
    assert not h.value
    assert L.moe_pipeline_submit(None, 1, None, None, None, 0, None, None, None, None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_pipeline_destroy(None) == moe.MOE_OK


def _header_prototypes():
    """name -> list of parameter type strings, from every MOE_API prototype in moe.h."""
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
    protos = {}
    for m in re.finditer(r"MOE_API\s+[\w\s\*]+?\b(moe_\w+)\s*\(([^)]*)\)\s*;", src):
        params = [p.strip() for p in m.group(2).split(",") if p.strip() and p.strip() != "void"]
        # drop the parameter name, keep the type
        protos[m.group(1)] = [re.sub(r"\b\w+\s*$", "", p).strip() for p in params]
    return protos


def _ctypes_kind(t):
    if t is ctypes.c_void_p or (isinstance(t, type) and issubclass(t, ctypes._Pointer)):
        return "ptr"
    return {ctypes.c_int32: "int32_t", ctypes.c_int64: "int64_t", ctypes.c_size_t: "size_t",
            ctypes.c_float: "float"}[t]


def _c_kind(t):
    if "*" in t or t in ("moe_stream_t",):
        return "ptr"
    return {"int32_t": "int32_t", "int64_t": "int64_t", "size_t": "size_t", "float": "float"}[t]


def test_binding_signatures_match_the_header():
    # every entry point the binding calls: same parameter count, and the same width for
    # every scalar (an int64 size passed as int32 would corrupt the call silently)
    from fp8_gemm_sigmoid_b300 import moe as m
    protos = _header_prototypes()
    assert set(m._SIGS) <= set(protos), set(m._SIGS) - set(protos)
    for name, sig in m._SIGS.items():
        c = [_c_kind(t) for t in protos[name]]
        py = [_ctypes_kind(t) for t in sig]
        assert c == py, (name, c, py)


def test_binding_constants_match_the_header():
    # the status codes, modes, epilogues and the fused-gate threshold the binding mirrors
    from fp8_gemm_sigmoid_b300 import moe as m
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    values = {k: int(v) for k, v in re.findall(r"\b(MOE_[A-Z0-9_]+)\s*=\s*(\d+)", src)}
    values.update({k: int(v) for k, v in re.findall(r"#define\s+(MOE_[A-Z0-9_]+)\s+(\d+)", src)})
    names = ["MOE_OK", "MOE_ERR_INVALID_ARG", "MOE_ERR_UNSUPPORTED", "MOE_ERR_WORKSPACE", "MOE_ERR_CUDA",
             "MOE_ERR_TIMEOUT", "MOE_FP32", "MOE_FP8_BLOCK", "MOE_MXFP8", "MOE_EPI_SWIGLU_QUANT", "MOE_EPI_STORE",
             "MOE_GATE_QUANT_MIN_TOKENS"]
    for n in names:
        assert values[n] == getattr(m, n), n


def test_more_host_side_rejections(moe):
    # every case below is refused before any CUDA call, so it runs without a GPU
    L = moe._lib_handle()
    vp, i64 = ctypes.c_void_p, ctypes.c_int64
    from fp8_gemm_sigmoid_b300 import synthetic as sy
    cfg = moe.make_config(sy.config("v3_prefill"))
    bad_cfg = moe.make_config(dict(sy.config("v3_prefill"), n_group=7))
    c, cb = ctypes.byref(cfg), ctypes.byref(bad_cfg)
    INV = moe.MOE_ERR_INVALID_ARG
    # gate
    assert L.moe_gate(c, -1, vp(16), vp(16), vp(16), vp(16), vp(16), vp(16), None) == INV
    assert L.moe_gate(c, 8, vp(16), vp(16), vp(16), vp(16), vp(16), None, None) == INV
    assert L.moe_gate(cb, 8, vp(16), vp(16), vp(16), vp(16), vp(16), vp(16), None) == INV
    assert L.moe_gate(c, 8, None, vp(16), vp(16), vp(16), vp(16), vp(16), None) == INV
    # combine: T == 0 enqueues nothing and succeeds; missing or misaligned buffers are refused;
    # the shared expert's rows are required exactly when the layer has a shared expert
    assert L.moe_combine(c, 0, None, None, None, None, None, None) == moe.MOE_OK
    assert L.moe_combine(c, 8, None, vp(16), vp(16), vp(16), vp(16), None) == INV
    assert L.moe_combine(c, 8, vp(16), vp(16), vp(16), vp(16), vp(24), None) == INV
    assert L.moe_combine(c, 8, vp(16), vp(16), vp(16), None, vp(16), None) == INV
    assert L.moe_combine(c, 8, vp(16), vp(16), vp(16), vp(24), vp(16), None) == INV
    no_shared = moe.make_config(dict(sy.config("v3_prefill"), has_shared=0))
    assert L.moe_combine(ctypes.byref(no_shared), 8, vp(16), vp(16), vp(16), vp(16), vp(16), None) == INV
    # bias update
    assert L.moe_bias_update(c, 8, vp(16), None, None) == INV
    assert L.moe_bias_update(c, -1, vp(16), vp(16), None) == INV
    # whole layer: missing weights, a misaligned or short workspace
    need = ctypes.c_size_t(0)
    assert L.moe_workspace_size(c, 64, ctypes.byref(need)) == moe.MOE_OK
    w = moe.moe_weights(vp(16), vp(16), vp(16), vp(16), vp(16))
    w_missing = moe.moe_weights(vp(16), None, vp(16), vp(16), vp(16))
    args = lambda ww, ws, nb: (c, 64, vp(16), ctypes.byref(ww), vp(16), 0, vp(16), vp(16), vp(16),  # noqa: E731
                               vp(16), ws, nb, None)
    assert L.moe_forward(*args(w_missing, vp(1024), need.value)) == INV
    assert L.moe_forward(*args(w, vp(1032 + 1), need.value)) == INV
    assert L.moe_forward(*args(w, vp(1024), need.value - 1)) == moe.MOE_ERR_WORKSPACE
    # the no-allocation permutation: beyond its fixed scratch (2 * ceil(T/64) * E > 2^20)
    f = L.moe_permute_noalloc
    f.argtypes = [moe._cfgp, i64, vp, vp, vp, vp, vp, vp, vp, vp, vp]
    f.restype = ctypes.c_int
    assert f(c, 200000, vp(16), vp(16), vp(16), vp(16), vp(16), vp(16), vp(16), vp(16), None) \
        == moe.MOE_ERR_UNSUPPORTED
    assert f(c, 100, vp(16), vp(16), vp(16), None, vp(16), vp(16), vp(16), vp(16), None) == INV
    assert f(c, 100, vp(16), vp(17), vp(16), vp(16), vp(16), vp(16), vp(16), vp(16), None) == INV
    # the bounded-wait self-test refuses budgets outside 1 .. 4e9 cycles
    assert L.moe_selftest_wait_timeout(0, None) == INV
    assert L.moe_selftest_wait_timeout(4000000001, None) == INV
    assert L.moe_device_error(None) == INV


def test_gate_quant_host_side_rejections(moe):
    # refused (INVALID_ARG) or declined (UNSUPPORTED) before any CUDA call, so no GPU is needed
    L = moe._lib_handle()
    vp = ctypes.c_void_p
    from fp8_gemm_sigmoid_b300 import synthetic as sy
    INV, UNS = moe.MOE_ERR_INVALID_ARG, moe.MOE_ERR_UNSUPPORTED
    cfg = lambda **kw: ctypes.byref(moe.make_config(dict(sy.config("v3_prefill"), **kw)))  # noqa: E731
    ok_args = (vp(16), vp(16), vp(16), vp(16), vp(16), vp(16), vp(16), vp(16), None)
    assert L.moe_gate_quant(cfg(), -1, *ok_args) == INV
    assert L.moe_gate_quant(cfg(), 8, vp(16), vp(16), vp(16), vp(16), vp(16), vp(16), None, vp(16), None) == INV
    assert L.moe_gate_quant(cfg(), 8, vp(16), vp(16), vp(16), vp(16), vp(16), vp(16), vp(16), None, None) == INV
    assert L.moe_gate_quant(cfg(n_group=7), 8, *ok_args) == INV
    # shapes outside the fused kernel: FP32 mode, groups of 16 experts, 288 experts
    assert L.moe_gate_quant(ctypes.byref(moe.make_config(sy.config("tiny_fp32"))), 8, *ok_args) == UNS
    assert L.moe_gate_quant(cfg(n_group=16, topk_group=4), 8, *ok_args) == UNS
    assert L.moe_gate_quant(cfg(n_experts=288, n_group=9, topk_group=2), 8, *ok_args) == UNS
    # misaligned x or codes
    assert L.moe_gate_quant(cfg(), 8, vp(24), vp(16), vp(16), vp(16), vp(16), vp(16), vp(16), vp(16), None) == UNS
    assert L.moe_gate_quant(cfg(), 8, vp(16), vp(16), vp(16), vp(16), vp(16), vp(16), vp(24), vp(16), None) == UNS


def test_logfmt_host_side_rejections(moe):
    L = moe._lib_handle()
    vp = ctypes.c_void_p
    INV = moe.MOE_ERR_INVALID_ARG
    for f in (L.moe_logfmt_encode, L.moe_logfmt_decode):
        assert f(8, 0, 128, None, None, None, None, None) == moe.MOE_OK  # no rows: nothing to do
        assert f(2, 4, 128, vp(16), vp(16), vp(16), vp(16), None) == INV  # n_bits below 3
        assert f(13, 4, 128, vp(16), vp(16), vp(16), vp(16), None) == INV  # above 12
        assert f(8, 4, 100, vp(16), vp(16), vp(16), vp(16), None) == INV   # cols not a multiple of 128
        assert f(8, -1, 128, vp(16), vp(16), vp(16), vp(16), None) == INV
        assert f(8, 4, 128, vp(16), vp(16), None, vp(16), None) == INV
        assert f(8, 4, 128, vp(24), vp(16), vp(16), vp(16), None) == INV  # misaligned
