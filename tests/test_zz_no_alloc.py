"""moe_expert_ffn_noalloc, the entry point for callers that cannot allocate device memory
(for example a plugin whose device memory belongs to its host runtime's pool): it must give
the same expert outputs as moe_expert_ffn with a caller-allocated workspace, call after call,
although every call reuses the library's one fixed scratch array.

This file is collected last on purpose, so that a run stopping at its first failure has
already run every other test. It also passes on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import moe_workloads as mw
import routed_expert_ffn_softmax_gb300 as moe

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
REL = {"bf16": 1e-2, "int8": 2e-2}  # the tolerance the parity tests use


@pytest.fixture(scope="module", autouse=True)
def _built():
    from routed_expert_ffn_softmax_gb300 import build
    build.build()
    moe.load()
    yield


def assert_close(got: torch.Tensor, ref: torch.Tensor, wtype: str, what: str):
    g = got.double().cpu().numpy()
    r = ref.double().cpu().numpy()
    assert np.all(np.isfinite(g)), f"{what}: non-finite output"
    bound = REL[wtype] * np.abs(r).max() + 1e-3
    err = np.abs(g - r).max()
    assert err <= bound, f"{what}: max err {err:.4g} > {bound:.4g}"


def routed_block(cfg, T, seed):
    """Routing and gathered token block from the library's own routing and gather."""
    L = {n: (v.to(DEV) if v is not None else None) for n, v in mw.make_layer(cfg, seed=seed).items()}
    x, lg = (t.to(DEV) for t in mw.make_tokens(cfg, T, seed=seed))
    k, P = cfg.top_k, T * cfg.top_k
    i32 = dict(dtype=torch.int32, device=DEV)
    r = dict(ids=torch.empty(T, k, **i32), w=torch.empty(T, k, device=DEV), counts=torch.empty(cfg.E, **i32),
             offsets=torch.empty(cfg.E + 1, **i32), st=torch.empty(P, **i32), inv=torch.empty(T, k, **i32),
             act=torch.empty(cfg.E, **i32), na=torch.empty(1, **i32))
    moe.moe_route_topk(lg, k, r["ids"], r["w"], r["counts"], r["offsets"], r["st"], r["inv"], r["act"], r["na"])
    xg = torch.empty(P, cfg.H, dtype=torch.bfloat16, device=DEV)
    moe.moe_gather(x, k, r["st"], xg)
    return L, r, xg


CASES = [
    # name, H, I, E, top_k, wtype, T    (split units across CTAs, ragged tails, several passes)
    ("bf16", 512, 1024, 8, 2, "bf16", 37),
    ("bf16_skew", 256, 512, 4, 2, "bf16", 150),
    ("int8", 384, 256, 8, 4, "int8", 70),
]


@pytest.mark.parametrize("name,H,I,E,k,wtype,T", CASES)
def test_noalloc_matches_workspace_entry_point_twice(name, H, I, E, k, wtype, T):
    cfg = mw.MoEConfig(name, H, I, E, k, wtype, (T,), skew_experts=(0, 1) if "skew" in name else (),
                       skew=3.0 if "skew" in name else 0.0)
    L, r, xg = routed_block(cfg, T, seed=H + T)
    P = T * k
    wt = moe.MOE_W_INT8_G128 if wtype == "int8" else moe.MOE_W_BF16
    ws = moe.alloc_workspace(T, H, I, E, k, wt, DEV)
    y_ref = torch.full((P, H), float("nan"), device=DEV)
    moe.moe_expert_ffn(xg, r["offsets"], r["act"], r["na"], L["W_gate"], L["W_up"], L["W_down"], L["s_gate"],
                       L["s_up"], L["s_down"], y_ref, ws)
    torch.cuda.synchronize()
    assert moe.workspace_status(ws) == 0
    for call in range(2):  # the second call reuses what the first left in the fixed scratch
        y = torch.full((P, H), float("nan"), device=DEV)
        moe.moe_expert_ffn_noalloc(xg, r["offsets"], r["act"], r["na"], L["W_gate"], L["W_up"], L["W_down"],
                                   L["s_gate"], L["s_up"], L["s_down"], y)
        torch.cuda.synchronize()
        assert_close(y, y_ref, wtype, f"{name} call {call + 1}")


def test_noalloc_rejects_blocks_larger_than_its_scratch():
    lib = moe.load()
    f = lib.moe_expert_ffn_noalloc
    V, i = ctypes.c_void_p, ctypes.c_int
    f.argtypes = [V, V, V, V, V, V, V, V, V, V, i, i, i, i, i, V, V]
    f.restype = i
    fake = 1 << 20  # aligned, never dereferenced: the size check comes first
    # P * I * 2 bytes = 2048 * 14336 * 2 = 56 MiB > the fixed scratch
    rc = f(fake, fake, fake, fake, fake, fake, fake, None, None, None, moe.MOE_W_BF16, 4096, 14336, 8, 2048,
           fake, None)
    assert rc == 3, moe.moe_status_string(rc)  # MOE_ERR_WORKSPACE, nothing launched
