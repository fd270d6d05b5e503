"""Residual-split INT8 experts on the GPU (moe_ffn_forward_residual / moe_expert_ffn_residual, through
the C ABI) against the residual-split oracle (needs a GPU).

RapidMoE (arXiv 2610.01265), "Residual-Split Representation": gate and up as W^Q + W^R (two INT8
streams summed before SiLU), down one INT8 copy. Tolerance: the INT8 bound,
|gpu - oracle| <= 2e-2 * max|oracle| + 1e-3 elementwise (identical dequantisation inputs).
"""
import numpy as np
import pytest
import torch

import moe_workloads as mw
import oracle
import routed_expert_ffn_softmax_gb300 as moe
from test_gpu_parity import DEV, assert_moe_close, check_route, gpu_route, to_np_f32

pytestmark = pytest.mark.gpu
RES = ("W_gate", "W_up", "W_down", "s_gate", "s_up", "s_down", "Wr_gate", "Wr_up", "sr_gate", "sr_up")


@pytest.fixture(scope="module", autouse=True)
def _built():
    from routed_expert_ffn_softmax_gb300 import build
    build.build()
    moe.load()
    yield


def case(T, H, I, E, k, seed, skew=()):
    cfg = mw.MoEConfig("res", H, I, E, k, "int8_residual", (T,), skew_experts=tuple(skew), skew=3.0 if skew else 0.0)
    L = mw.make_layer(cfg, seed=seed)
    x, lg = mw.make_tokens(cfg, T, seed=seed)
    return cfg, L, x, lg


def gpu_forward(L, x, lg, k):
    d = {n: L[n].to(DEV) for n in RES}
    T, H = x.shape
    E, I, _ = L["W_gate"].shape
    ws = moe.alloc_workspace(T, H, I, E, k, moe.MOE_W_INT8_G128, DEV)
    out = torch.full((T, H), float("nan"), dtype=torch.bfloat16, device=DEV)
    moe.moe_ffn_forward_residual(x.to(DEV), lg.to(DEV), *(d[n] for n in RES), k, out, ws)
    torch.cuda.synchronize()
    assert moe.workspace_status(ws) == 0
    return out


def oracle_forward(L, x, lg, k):
    return oracle.forward_residual(x, lg, L["W_gate"], L["s_gate"], L["Wr_gate"], L["sr_gate"], L["W_up"], L["s_up"],
                                   L["Wr_up"], L["sr_up"], L["W_down"], L["s_down"], top_k=k)


@pytest.mark.parametrize("T,H,I,E,k,skew", [
    (4, 256, 384, 8, 2, ()),
    (70, 384, 256, 8, 4, (2,)),        # skewed: one expert well past a 32-token pass
    (8, 640, 384, 64, 8, (5,)),        # one expert gets all 8 tokens, 56 others one each
    (33, 128, 512, 16, 2, ()),
])
def test_forward_matches_oracle(T, H, I, E, k, skew):
    cfg, L, x, lg = case(T, H, I, E, k, seed=T + H, skew=skew)
    out = gpu_forward(L, x, lg, k)
    ref = oracle_forward(L, x, lg, k)
    assert_moe_close(to_np_f32(out), oracle.bf16_bits_to_f32(ref["out"]), "int8", f"residual T={T} H={H} I={I}")


def test_expert_ffn_entry_point_matches_oracle():
    """route -> gather -> moe_expert_ffn_residual -> combine as separate calls; Y against the oracle's
    per-assignment expert outputs."""
    T, H, I, E, k = 12, 256, 256, 16, 4
    cfg, L, x, lg = case(T, H, I, E, k, seed=21)
    d = {n: L[n].to(DEV) for n in RES}
    P = T * k
    i32 = dict(dtype=torch.int32, device=DEV)
    r = dict(ids=torch.empty(T, k, **i32), w=torch.empty(T, k, device=DEV), counts=torch.empty(E, **i32),
             offsets=torch.empty(E + 1, **i32), sorted_token=torch.empty(P, **i32), inv_pos=torch.empty(T, k, **i32),
             active=torch.empty(E, **i32), num_active=torch.empty(1, **i32))
    moe.moe_route_topk(lg.to(DEV), k, r["ids"], r["w"], r["counts"], r["offsets"], r["sorted_token"], r["inv_pos"],
                       r["active"], r["num_active"])
    xg = torch.empty(P, H, dtype=torch.bfloat16, device=DEV)
    moe.moe_gather(x.to(DEV), k, r["sorted_token"], xg)
    Y = torch.full((P, H), float("nan"), dtype=torch.float32, device=DEV)
    ws = moe.alloc_workspace(T, H, I, E, k, moe.MOE_W_INT8_G128, DEV)
    moe.moe_expert_ffn_residual(xg, r["offsets"], r["active"], r["num_active"], *(d[n] for n in RES), Y, ws)
    torch.cuda.synchronize()
    assert moe.workspace_status(ws) == 0
    ro = oracle.route(lg, k)
    Yg = Y.cpu().numpy()
    for t in range(T):
        for j in range(k):
            e = int(ro["ids"][t, j])
            h, _, _ = oracle.gateup_token_residual(x[t], L["W_gate"][e], L["s_gate"][e], L["Wr_gate"][e],
                                                   L["sr_gate"][e], L["W_up"][e], L["s_up"][e], L["Wr_up"][e],
                                                   L["sr_up"][e])
            y = oracle.down_token(h, L["W_down"][e], L["s_down"][e], "int8")
            assert_moe_close(Yg[int(ro["inv_pos"][t, j])], y, "int8", f"Y row of token {t} slot {j}")


def test_residual_reaches_below_int8_error():
    """On the GPU, as in the oracle, the split's gate/up error against the unquantised weights is far
    below INT8's: compare whole-FFN outputs against the BF16 oracle on the unquantised draws at the
    GPU's own precision (the residual result must be closer than the INT8 one)."""
    T, H, I, E, k = 16, 512, 512, 8, 2
    cfg, L, x, lg = case(T, H, I, E, k, seed=30)
    import dataclasses
    bf = mw.make_layer(dataclasses.replace(cfg, wtype="bf16"), seed=30)
    ref = oracle.forward(x, lg, bf["W_gate"], bf["W_up"], bf["W_down"], wtype="bf16", top_k=k)["out_f32"]
    res = to_np_f32(gpu_forward(L, x, lg, k))
    d = {n: L[n].to(DEV) for n in RES}
    ws = moe.alloc_workspace(T, H, I, E, k, moe.MOE_W_INT8_G128, DEV)
    out8 = torch.empty(T, H, dtype=torch.bfloat16, device=DEV)
    moe.moe_ffn_forward(x.to(DEV), lg.to(DEV), d["W_gate"], d["W_up"], d["W_down"], d["s_gate"], d["s_up"],
                        d["s_down"], k, out8, ws)
    torch.cuda.synchronize()
    i8 = to_np_f32(out8)
    assert np.abs(res - ref).mean() < np.abs(i8 - ref).mean()


@pytest.mark.parametrize("T", [1, 8, 64, 256])
def test_full_size_every_token(T):
    cfg = mw.CONFIGS["qwen3_int8_residual"]
    Lg = mw.make_layer(cfg, device=DEV)
    x, lg = mw.make_tokens(cfg, T, device=DEV)
    ws = moe.alloc_workspace(T, cfg.H, cfg.I, cfg.E, cfg.top_k, moe.MOE_W_INT8_G128, DEV)
    out = torch.full((T, cfg.H), float("nan"), dtype=torch.bfloat16, device=DEV)
    moe.moe_ffn_forward_residual(x, lg, *(Lg[n] for n in RES), cfg.top_k, out, ws)
    torch.cuda.synchronize()
    assert moe.workspace_status(ws) == 0
    got = to_np_f32(out)
    assert np.all(np.isfinite(got))
    ro = oracle.route(lg.cpu(), cfg.top_k)
    check_route(gpu_route(lg, cfg.top_k), ro)
    Lc = {n: Lg[n].cpu() for n in RES}
    xc = x.cpu()
    for t in range(T):
        ys = []
        for j in range(cfg.top_k):
            e = int(ro["ids"][t, j])
            W = {n: Lc[n][e] for n in RES}
            h, _, _ = oracle.gateup_token_residual(xc[t], W["W_gate"], W["s_gate"], W["Wr_gate"], W["sr_gate"],
                                                   W["W_up"], W["s_up"], W["Wr_up"], W["sr_up"])
            ys.append(oracle.down_token(h, W["W_down"], W["s_down"], "int8"))
        row, _ = oracle.combine_token(np.stack(ys), ro["w"][t])
        assert_moe_close(got[t], oracle.bf16_bits_to_f32(row), "int8", f"residual full size T={T} token {t}")
    del Lg, Lc
    torch.cuda.empty_cache()
