"""moe_permute_noalloc: the permutation for callers that cannot allocate device memory or pass
a workspace (frameworks that own the whole memory budget, loops that cannot afford
cudaMalloc's device synchronisation, plugin signatures with only inputs and outputs).

Called through the C ABI, it must give exactly what moe_permute (the workspace version)
gives -- the permutation is integer and byte work, so the tolerance is bit-exactness -- on
two calls in a row with different inputs (the shared static scratch keeps the previous
call's contents, which must not leak into the next one).  Collected last so that a run that
stops at the first failure has already run every other test; it also passes alone."""
import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module")
def moe():
    from fp8_gemm_sigmoid_b300 import build, moe as m
    build.build()
    assert torch.cuda.is_available()
    return m


def _case(T, E, K, S, seed):
    rng = np.random.default_rng(seed)
    p = rng.dirichlet(np.full(E, 0.5))
    idx = np.stack([rng.choice(E, K, replace=False, p=p) for _ in range(T)]).astype(np.int32)
    cfg = dict(hidden=512, inter=256, n_experts=E, n_group=8, topk_group=4, top_k=K,
               routed_scaling_factor=2.5, has_shared=S, mode="fp8")
    g = torch.Generator(device=DEV).manual_seed(seed)
    xq = torch.randint(0, 255, (T, 512), generator=g, device=DEV, dtype=torch.uint8)
    xs = torch.rand(T, 4, generator=g, device=DEV)
    return cfg, torch.from_numpy(idx).to(DEV), xq, xs


def _outputs(cfg, T):
    E, K, S = cfg["n_experts"], cfg["top_k"], cfg["has_shared"]
    R = T * K + T * S
    return dict(offs=torch.full((E + 1 + S,), -1, dtype=torch.int32, device=DEV),
                perm_tok=torch.full((R,), -1, dtype=torch.int32, device=DEV),
                row_of=torch.full((T, K), -1, dtype=torch.int32, device=DEV),
                aq=torch.zeros(R, 512, dtype=torch.uint8, device=DEV),
                as_=torch.zeros(4, R, dtype=torch.float32, device=DEV))  # K-block-major


def test_noalloc_matches_workspace_permute_on_two_calls(moe):
    for T, E, K, S, seed in [(3001, 256, 8, 1, 1), (700, 64, 4, 0, 2)]:
        cfg, idx, xq, xs = _case(T, E, K, S, seed)
        ref = _outputs(cfg, T)
        counts = torch.bincount(idx.view(-1).long(), minlength=E).to(torch.int32)
        ws = moe.workspace(cfg, T)
        moe.moe_permute(cfg, T, idx, counts, xq, xs, ref["offs"], ref["perm_tok"], ref["row_of"],
                        ref["aq"], ref["as_"], ws)
        got = _outputs(cfg, T)
        moe.moe_permute_noalloc(cfg, T, idx, xq, xs, got["offs"], got["perm_tok"], got["row_of"],
                                got["aq"], got["as_"])
        torch.cuda.synchronize()
        for k in ref:
            assert torch.equal(got[k], ref[k]), (T, k)


def test_noalloc_rejects_sizes_beyond_its_scratch(moe):
    # 2 * ceil(T/64) * E int32 must fit the 4 MiB array: E = 1024 allows T <= 32768
    cfg = moe.make_config(dict(hidden=512, inter=256, n_experts=1024, n_group=32, topk_group=4,
                               top_k=8, routed_scaling_factor=1.0, has_shared=0, mode="fp8"))
    L = moe._lib_handle()
    f = L.moe_permute_noalloc
    vp = ctypes.c_void_p
    f.argtypes = [ctypes.POINTER(moe.moe_config), ctypes.c_int64] + [vp] * 9
    f.restype = ctypes.c_int
    args = [vp(256)] * 8
    assert f(ctypes.byref(cfg), 32768 + 64, *args, None) == moe.MOE_ERR_UNSUPPORTED
