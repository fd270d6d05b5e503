"""Pins of the residual-split oracle to things other than itself (no GPU).

RapidMoE (arXiv 2610.01265), "Residual-Split Representation" and "GLU Architecture Adoption":
W^H = W^Q + W^R, with gate/up computed as W^Q x + W^R x before SiLU and down kept as one separate
copy. The oracle (moe_oracle.cpp) dequantises w = qQ * sQ + qR * sR. Pins: the split quantiser's
error bound; a zero residual reduces exactly to the INT8 oracle and a zero low part exactly to the
BF16 oracle (power-of-two scales make the dequantised weights bf16 values); gate/up
preactivations are the sum of the two parts' (linearity, the decomposition the pages build on);
and the split is closer to the unquantised FFN than INT8 alone.
"""
import dataclasses

import numpy as np
import torch

import moe_workloads as mw
import oracle


def case(T=5, H=256, I=384, E=8, k=2, seed=3):
    cfg = mw.MoEConfig("res", H, I, E, k, "int8_residual", (T,))
    L = mw.make_layer(cfg, seed=seed)
    x, lg = mw.make_tokens(cfg, T, seed=seed)
    return cfg, L, x, lg


def fwd_res(x, lg, L, k):
    return oracle.forward_residual(x, lg, L["W_gate"], L["s_gate"], L["Wr_gate"], L["sr_gate"], L["W_up"],
                                   L["s_up"], L["Wr_up"], L["sr_up"], L["W_down"], L["s_down"], top_k=k)


def test_split_quantiser_error_bound():
    w = mw.draw_weights(4, 96, 512, seed=1, tensor=2)
    qQ, sQ, qR, sR = mw.quantize_int8_residual(w)
    g = lambda q, s: (q.float().reshape(4, 96, 4, 128) * s[..., None]).reshape(4, 96, 512)
    err = (g(qQ, sQ) + g(qR, sR) - w.float()).abs().reshape(4, 96, 4, 128)
    # half a residual step, plus the fp32 rounding of adding up terms of magnitude |w| (4 ulps)
    ulps = 4 * 2.0 ** -23 * w.float().abs().reshape(4, 96, 4, 128)
    assert torch.all(err <= sR[..., None] * 0.5 + ulps)
    # the residual is at most half a step of W^Q, so its scale is at most 1/254 of W^Q's (up to the
    # fp32 error of w / sQ near a rounding tie: 2 * 127 * 2^-24 of sQ, i.e. a factor 1 + 3e-5)
    assert torch.all(sR <= sQ / 254 * (1 + 3.1e-5))
    # INT8 alone errs by up to half of its own (254x coarser) step
    assert (g(qQ, sQ) - w.float()).abs().max() > 50 * err.max()


def test_zero_residual_is_the_int8_oracle():
    cfg, L, x, lg = case()
    L = dict(L, Wr_gate=torch.zeros_like(L["Wr_gate"]), Wr_up=torch.zeros_like(L["Wr_up"]))
    got = fwd_res(x, lg, L, cfg.top_k)
    ref = oracle.forward(x, lg, L["W_gate"], L["W_up"], L["W_down"], L["s_gate"], L["s_up"], L["s_down"],
                         wtype="int8", top_k=cfg.top_k)
    assert np.array_equal(got["out"], ref["out"]) and np.array_equal(got["out_f32"], ref["out_f32"])


def test_zero_low_part_is_the_bf16_oracle():
    """qQ = 0 and power-of-two residual and down scales: every dequantised weight is a bf16 value,
    so the BF16 oracle on those weights must agree bit for bit."""
    cfg, L, x, lg = case(seed=9)
    g = torch.Generator().manual_seed(4)
    pow2 = lambda s: torch.exp2(torch.randint(-12, -6, s.shape, generator=g).float())
    L = dict(L)
    L["W_gate"] = torch.zeros_like(L["W_gate"])
    L["W_up"] = torch.zeros_like(L["W_up"])
    for n in ("sr_gate", "sr_up", "s_down"):
        L[n] = pow2(L[n])
    deq = lambda q, s: (q.float().reshape(*q.shape[:-1], -1, 128) * s[..., None]).reshape(q.shape)
    Wg = deq(L["Wr_gate"], L["sr_gate"]).to(torch.bfloat16)
    Wu = deq(L["Wr_up"], L["sr_up"]).to(torch.bfloat16)
    Wd = deq(L["W_down"], L["s_down"]).to(torch.bfloat16)
    assert torch.equal(Wg.float(), deq(L["Wr_gate"], L["sr_gate"]))  # exact in bf16
    got = fwd_res(x, lg, L, cfg.top_k)
    ref = oracle.forward(x, lg, Wg, Wu, Wd, wtype="bf16", top_k=cfg.top_k)
    assert np.array_equal(got["out"], ref["out"]) and np.array_equal(got["out_f32"], ref["out_f32"])


def test_preactivations_are_linear_in_the_split():
    cfg, L, x, lg = case(seed=5)
    e = 3
    _, g_res, u_res = oracle.gateup_token_residual(x[0], L["W_gate"][e], L["s_gate"][e], L["Wr_gate"][e],
                                                   L["sr_gate"][e], L["W_up"][e], L["s_up"][e], L["Wr_up"][e],
                                                   L["sr_up"][e])
    _, gq, uq = oracle.gateup_token(x[0], L["W_gate"][e], L["W_up"][e], L["s_gate"][e], L["s_up"][e], "int8")
    _, gr, ur = oracle.gateup_token(x[0], L["Wr_gate"][e], L["Wr_up"][e], L["sr_gate"][e], L["sr_up"][e], "int8")
    mag = np.abs(x[0].float().numpy()).sum() * 0.1  # bound on sum |x w| for these weights
    np.testing.assert_allclose(g_res, gq + gr, rtol=0, atol=1e-5 * mag)
    np.testing.assert_allclose(u_res, uq + ur, rtol=0, atol=1e-5 * mag)


def test_split_gate_up_is_closer_to_the_unquantised_weights():
    """The split's purpose: gate/up preactivations with W^Q + W^R track the unquantised weights far
    more closely than with W^Q alone (down is not split, so the whole FFN gains less)."""
    cfg, L, x, lg = case(T=6, seed=12)
    bf = mw.make_layer(dataclasses.replace(cfg, wtype="bf16"), seed=12)  # the same draws, unquantised
    e = 5
    _, g_ref, u_ref = oracle.gateup_token(x[1], bf["W_gate"][e], bf["W_up"][e], wtype="bf16")
    _, g_res, u_res = oracle.gateup_token_residual(x[1], L["W_gate"][e], L["s_gate"][e], L["Wr_gate"][e],
                                                   L["sr_gate"][e], L["W_up"][e], L["s_up"][e], L["Wr_up"][e],
                                                   L["sr_up"][e])
    _, g_i8, u_i8 = oracle.gateup_token(x[1], L["W_gate"][e], L["W_up"][e], L["s_gate"][e], L["s_up"][e], "int8")
    for ref, res, i8 in ((g_ref, g_res, g_i8), (u_ref, u_res, u_i8)):
        assert np.abs(res - ref).mean() < 0.05 * np.abs(i8 - ref).mean()
