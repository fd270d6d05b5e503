"""moe_expert_ffn_noalloc, the entry point for callers that cannot allocate device memory (for
example a plugin whose device memory belongs to its host runtime's pool, or a decode loop that must
not call cudaMalloc mid-step): every call reuses the library's one fixed scratch array, yet each of
two calls in a row must give the oracle's expert outputs, leave the scratch's status word at 0 (read
back through moe_expert_ffn_noalloc_status) and agree with moe_expert_ffn and its caller-allocated
workspace.

This file is collected last on purpose, so that a run stopping at its first failure has already run
every other test. It also passes on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import moe_workloads as mw
import oracle
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


def assert_close(got, ref, wtype: str, what: str):
    g = np.asarray(got, np.float64)
    r = np.asarray(ref, np.float64)
    assert np.all(np.isfinite(g)), f"{what}: non-finite output"
    bound = REL[wtype] * np.abs(r).max() + 1e-3
    err = np.abs(g - r).max()
    assert err <= bound, f"{what}: max err {err:.4g} > {bound:.4g}"


def routed_block(cfg, T, seed):
    """Layer (CPU and device), routing and gathered token block from the library's own routing and gather."""
    Lc = mw.make_layer(cfg, seed=seed)
    L = {n: (v.to(DEV) if v is not None else None) for n, v in Lc.items()}
    x, lg = mw.make_tokens(cfg, T, seed=seed)
    k, P = cfg.top_k, T * cfg.top_k
    i32 = dict(dtype=torch.int32, device=DEV)
    r = dict(ids=torch.empty(T, k, **i32), w=torch.empty(T, k, device=DEV), counts=torch.empty(cfg.E, **i32),
             offsets=torch.empty(cfg.E + 1, **i32), st=torch.empty(P, **i32), inv=torch.empty(T, k, **i32),
             act=torch.empty(cfg.E, **i32), na=torch.empty(1, **i32))
    moe.moe_route_topk(lg.to(DEV), k, r["ids"], r["w"], r["counts"], r["offsets"], r["st"], r["inv"], r["act"],
                       r["na"])
    xg = torch.empty(P, cfg.H, dtype=torch.bfloat16, device=DEV)
    moe.moe_gather(x.to(DEV), k, r["st"], xg)
    return Lc, L, x, lg, r, xg


def oracle_expert_rows(cfg, Lc, x, lg):
    """The oracle's expert output y for every assignment, in the expert-sorted order of the block."""
    ro = oracle.route(lg, cfg.top_k)
    T = x.shape[0]
    Y = np.zeros((T * cfg.top_k, cfg.H), np.float32)
    for t in range(T):
        for j in range(cfg.top_k):
            e = int(ro["ids"][t, j])
            sc = (lambda n: Lc[n][e] if Lc[n] is not None else None)
            h, _, _ = oracle.gateup_token(x[t], Lc["W_gate"][e], Lc["W_up"][e], sc("s_gate"), sc("s_up"), cfg.wtype)
            Y[ro["inv_pos"][t, j]] = oracle.down_token(h, Lc["W_down"][e], sc("s_down"), cfg.wtype)
    return Y


CASES = [
    # name, H, I, E, top_k, wtype, T    (split units across CTAs, ragged tails, several passes)
    ("bf16", 512, 1024, 8, 2, "bf16", 37),
    ("bf16_skew", 256, 512, 4, 2, "bf16", 150),
    ("int8", 384, 256, 8, 4, "int8", 70),
]


@pytest.mark.parametrize("name,H,I,E,k,wtype,T", CASES)
def test_noalloc_matches_oracle_twice(name, H, I, E, k, wtype, T):
    cfg = mw.MoEConfig(name, H, I, E, k, wtype, (T,), skew_experts=(0, 1) if "skew" in name else (),
                       skew=3.0 if "skew" in name else 0.0)
    Lc, L, x, lg, r, xg = routed_block(cfg, T, seed=H + T)
    P = T * k
    ref = oracle_expert_rows(cfg, Lc, x, lg)
    wt = moe.MOE_W_INT8_G128 if wtype == "int8" else moe.MOE_W_BF16
    ws = moe.alloc_workspace(T, H, I, E, k, wt, DEV)
    y_ws = torch.full((P, H), float("nan"), device=DEV)
    moe.moe_expert_ffn(xg, r["offsets"], r["act"], r["na"], L["W_gate"], L["W_up"], L["W_down"], L["s_gate"],
                       L["s_up"], L["s_down"], y_ws, ws)
    torch.cuda.synchronize()
    assert moe.workspace_status(ws) == 0
    for call in range(2):  # the second call reuses what the first left in the fixed scratch
        y = torch.full((P, H), float("nan"), device=DEV)
        moe.moe_expert_ffn_noalloc(xg, r["offsets"], r["act"], r["na"], L["W_gate"], L["W_up"], L["W_down"],
                                   L["s_gate"], L["s_up"], L["s_down"], y)
        assert moe.moe_expert_ffn_noalloc_status() == 0, f"{name} call {call + 1}: a kernel gave up a wait"
        got = y.cpu().numpy()
        for p in range(P):
            assert_close(got[p], ref[p], wtype, f"{name} call {call + 1} row {p}")
        assert_close(got, y_ws.cpu().numpy(), wtype, f"{name} call {call + 1} vs moe_expert_ffn")


def test_noalloc_rejects_blocks_larger_than_its_scratch():
    """P * I * 2 bytes = 2048 * 14336 * 2 = 56 MiB of intermediate exceed the fixed scratch: the call
    must return MOE_ERR_WORKSPACE before launching anything. Every pointer is a real (small) device
    tensor, aligned and non-null, so the argument checks pass and only the size check rejects."""
    lib = moe.load()
    f = lib.moe_expert_ffn_noalloc
    V, i = ctypes.c_void_p, ctypes.c_int
    f.argtypes = [V, V, V, V, V, V, V, V, V, V, i, i, i, i, i, V, V]
    f.restype = i
    bufs = [torch.zeros(64, dtype=torch.int32, device=DEV) for _ in range(8)]
    p = [b.data_ptr() for b in bufs]
    rc = f(p[0], p[1], p[2], p[3], p[4], p[5], p[6], None, None, None, moe.MOE_W_BF16, 4096, 14336, 8, 2048,
           p[7], None)
    torch.cuda.synchronize()
    assert rc == 3, moe.moe_status_string(rc)  # MOE_ERR_WORKSPACE, nothing launched
    assert all(not b.any() for b in bufs)     # nothing was written
