"""Pins of the CPU oracle to things other than itself (no GPU).

Each test checks the oracle against a fact the pages or the mathematics fix:
hand-worked fixtures, a float64 brute force written independently (dense over
all experts with masked routing weights), closed forms (identity weights,
x = 0, top_k = 1, top_k = E), invariants (identical experts, token
permutation) and an exact INT8 / BF16 equivalence under power-of-two scales.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import moe_workloads as mw
import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def f64_to_bf16_value(v: np.ndarray) -> np.ndarray:
    """Round float64 values to the nearest bf16 value (ties to even), returned as float64."""
    v = np.asarray(v, dtype=np.float64)
    m, e = np.frexp(v)                     # v = m * 2**e, 0.5 <= |m| < 1
    r = np.rint(m * 256.0) / 256.0         # 8 significant bits, half to even
    return np.ldexp(r, e)


def bf16_ulp(v: np.ndarray) -> np.ndarray:
    v = np.abs(np.asarray(v, dtype=np.float64))
    _, e = np.frexp(np.where(v == 0, 1.0, v))
    return np.ldexp(1.0, e - 8)


# ----------------------------------------------------------------------------
# independent float64 brute force
def brute_route(logits: np.ndarray, k: int):
    T, E = logits.shape
    ids = np.zeros((T, k), np.int64)
    w = np.zeros((T, k), np.float64)
    for t in range(T):
        l = logits[t].astype(np.float64)
        order = np.lexsort((np.arange(E), -l))  # primary: -logit, secondary: id
        sel = order[:k]
        ex = np.exp(l[sel] - l[sel].max())
        ids[t] = sel
        w[t] = ex / ex.sum()
    return ids, w


def brute_sort(ids: np.ndarray, E: int):
    """Naive O(P*E) scan: per expert, the tokens that chose it in ascending order."""
    T, k = ids.shape
    counts = np.array([int((ids == e).sum()) for e in range(E)])
    offsets = np.concatenate([[0], np.cumsum(counts)])
    sorted_token = []
    for e in range(E):
        sorted_token += [t for t in range(T) if e in ids[t]]
    inv = np.zeros((T, k), np.int64)
    for t in range(T):
        for j in range(k):
            e = ids[t, j]
            toks = [tt for tt in range(T) if e in ids[tt]]
            inv[t, j] = offsets[e] + toks.index(t)
    active = np.array([e for e in range(E) if counts[e] > 0])
    return counts, offsets, np.array(sorted_token), inv, active


def dequant64(W, s):
    """int8 q [E,R,K] + scales [E,R,K/128] -> float64 weights; bf16 -> float64 if s is None."""
    if s is None:
        return W.float().double().numpy()
    q = W.double().numpy()
    sc = np.repeat(s.double().numpy(), 128, axis=-1)
    return q * sc


def brute_forward64(x, logits, Wg, Wu, Wd, k, sg=None, su=None, sd=None):
    """Dense over every expert with masked routing weights, float64 throughout; h rounded to bf16."""
    x64 = x.float().double().numpy()
    lg = logits.numpy()
    T = x64.shape[0]
    E = Wg.shape[0]
    wg, wu, wd = dequant64(Wg, sg), dequant64(Wu, su), dequant64(Wd, sd)
    ids, w = brute_route(lg, k)
    mask = np.zeros((T, E))
    for t in range(T):
        mask[t, ids[t]] = w[t]
    g = np.einsum("th,eih->tei", x64, wg)
    u = np.einsum("th,eih->tei", x64, wu)
    h = f64_to_bf16_value(g / (1.0 + np.exp(-g)) * u)
    y = np.einsum("tei,ehi->teh", h, wd)
    out = np.einsum("te,teh->th", mask, y)
    return dict(ids=ids, w=w, h=h, y=y, out=out, wd=wd)


# ----------------------------------------------------------------------------
# routing
@pytest.mark.parametrize("T,E,k,seed", [(1, 8, 2, 0), (7, 8, 2, 1), (16, 64, 8, 2), (33, 256, 8, 3),
                                        (5, 5, 5, 4), (9, 128, 1, 5)])
def test_route_matches_brute_force(T, E, k, seed):
    g = torch.Generator().manual_seed(seed)
    lg = torch.randn(T, E, generator=g)
    r = oracle.route(lg, k)
    ids, w = brute_route(lg.numpy(), k)
    np.testing.assert_array_equal(r["ids"], ids)
    np.testing.assert_allclose(r["w"], w, rtol=1e-6, atol=1e-7)
    counts, offsets, st, inv, active = brute_sort(ids, E)
    np.testing.assert_array_equal(r["counts"], counts)
    np.testing.assert_array_equal(r["offsets"], offsets)
    np.testing.assert_array_equal(r["sorted_token"], st)
    np.testing.assert_array_equal(r["inv_pos"], inv)
    np.testing.assert_array_equal(r["active"], active)


def test_route_ties_lower_id_first():
    g = torch.Generator().manual_seed(11)
    lg = torch.randint(-2, 3, (40, 16), generator=g).float()  # many exact ties
    r = oracle.route(lg, 4)
    ids, _ = brute_route(lg.numpy(), 4)
    np.testing.assert_array_equal(r["ids"], ids)


def test_route_golden_worked_cases():
    with open(os.path.join(GOLDEN, "routing_worked.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        lg = torch.tensor(c["logits"], dtype=torch.float32)
        r = oracle.route(lg, c["top_k"])
        np.testing.assert_array_equal(r["ids"], np.array(c["ids"]), err_msg=c["name"])
        if "w" in c:
            if c["w_exact"]:
                np.testing.assert_array_equal(r["w"], np.array(c["w"], np.float32), err_msg=c["name"])
            else:
                np.testing.assert_allclose(r["w"], np.array(c["w"]), rtol=1e-6, err_msg=c["name"])
        for key in ("counts", "offsets", "sorted_token", "inv_pos", "active"):
            if key in c:
                np.testing.assert_array_equal(r[key], np.array(c[key]), err_msg=f"{c['name']}:{key}")


def test_route_top1_weight_is_exactly_one():
    lg = torch.randn(50, 32, generator=torch.Generator().manual_seed(3))
    r = oracle.route(lg, 1)
    assert np.all(r["w"] == np.float32(1.0))
    np.testing.assert_array_equal(r["ids"][:, 0], lg.numpy().argmax(axis=1))


def test_route_topk_equal_E_is_full_softmax():
    lg = torch.randn(20, 16, generator=torch.Generator().manual_seed(4))
    r = oracle.route(lg, 16)
    l64 = lg.double().numpy()
    sm = np.exp(l64 - l64.max(1, keepdims=True))
    sm /= sm.sum(1, keepdims=True)
    full = np.take_along_axis(sm, r["ids"].astype(np.int64), axis=1)
    np.testing.assert_allclose(r["w"], full, rtol=2e-6, atol=1e-8)
    np.testing.assert_allclose(r["w"].astype(np.float64).sum(1), 1.0, atol=2e-6)


def test_route_weights_sum_to_one_and_descend():
    lg = torch.randn(64, 256, generator=torch.Generator().manual_seed(5))
    r = oracle.route(lg, 8)
    np.testing.assert_allclose(r["w"].astype(np.float64).sum(1), 1.0, atol=1e-6)
    assert np.all(np.diff(r["w"], axis=1) <= 0)


# ----------------------------------------------------------------------------
# expert FFN
def _tiny_layer(E, H, I, seed, wtype="bf16"):
    cfg = mw.MoEConfig("t", H, I, E, 1, wtype, (1,))
    return mw.make_layer(cfg, seed=seed)


def test_swiglu_golden_worked_example():
    with open(os.path.join(GOLDEN, "swiglu_worked.json")) as f:
        c = json.load(f)
    bf = lambda a: torch.tensor(a, dtype=torch.float32).to(torch.bfloat16)
    x, Wg, Wu, Wd = bf(c["x"]), bf(c["W_gate"]), bf(c["W_up"]), bf(c["W_down"])
    h, gg, uu = oracle.gateup_token(x[0], Wg[0], Wu[0])
    np.testing.assert_array_equal(gg, np.array(c["g"], np.float32))
    np.testing.assert_array_equal(uu, np.array(c["u"], np.float32))
    np.testing.assert_array_equal(oracle.bf16_bits_to_f32(h), np.array(c["h_bf16"], np.float32))
    y = oracle.down_token(h, Wd[0])
    np.testing.assert_array_equal(y, np.array(c["y"], np.float32))
    r = oracle.forward(x, torch.tensor(c["logits"]), Wg, Wu, Wd, top_k=1)
    np.testing.assert_array_equal(oracle.bf16_bits_to_f32(r["out"]), np.array(c["out_bf16"], np.float32))


@pytest.mark.parametrize("E,H,I,T,k,seed", [(4, 32, 48, 3, 2, 0), (8, 64, 64, 8, 2, 1), (6, 16, 40, 5, 6, 2),
                                            (8, 48, 32, 7, 1, 3)])
def test_forward_matches_fp64_brute_force(E, H, I, T, k, seed):
    L = _tiny_layer(E, H, I, seed)
    gen = torch.Generator().manual_seed(100 + seed)
    x = torch.randn(T, H, generator=gen).to(torch.bfloat16)
    lg = torch.randn(T, E, generator=gen)
    r = oracle.forward(x, lg, L["W_gate"], L["W_up"], L["W_down"], top_k=k, intermediates=True)
    b = brute_forward64(x, lg, L["W_gate"], L["W_up"], L["W_down"], k)
    np.testing.assert_array_equal(r["ids"], b["ids"])
    # h: equal to the fp64 brute force rounded to bf16, except where fp32 accumulation
    # moved the value across a bf16 rounding boundary (then off by one bf16 ulp).
    h32 = oracle.bf16_bits_to_f32(r["h"]).astype(np.float64)           # [T,k,I]
    h64 = np.stack([b["h"][t, b["ids"][t]] for t in range(T)])           # [T,k,I]
    dh = np.abs(h32 - h64)
    assert np.all(dh <= bf16_ulp(np.maximum(np.abs(h32), np.abs(h64))) * 1.0001)
    assert (dh > 0).mean() < 0.02
    # y: fp64 y from the brute force's h; bound = flips * |Wd| + fp32 sequential-sum error.
    eps = 2.0 ** -24
    for t in range(T):
        for j in range(k):
            e = b["ids"][t, j]
            wd = b["wd"][e]                                              # [H,I]
            y64 = b["y"][t, e]
            bound = np.abs(wd) @ dh[t, j] + 1.01 * I * eps * (np.abs(wd) @ np.abs(h32[t, j])) + 1e-30
            assert np.all(np.abs(r["y"][t, j] - y64) <= bound), (t, j)
    # out (fp32 before the final rounding) vs the fp64 mixture
    ybound = np.zeros((T, H))
    for t in range(T):
        for j in range(k):
            e = b["ids"][t, j]
            ybound[t] += b["w"][t, j] * (np.abs(b["wd"][e]) @ dh[t, j]
                                         + 1.01 * I * eps * (np.abs(b["wd"][e]) @ np.abs(h32[t, j])))
    mag = np.einsum("tj,tjh->th", np.abs(b["w"]), np.abs(r["y"]).astype(np.float64))
    bound = ybound + 2e-6 * mag + (k + 1) * eps * mag + 1e-30
    assert np.all(np.abs(r["out_f32"] - b["out"]) <= bound)
    # out bits are the fp32 value rounded once to bf16
    np.testing.assert_array_equal(r["out"], oracle.f32_to_bf16_bits(r["out_f32"]))


def test_identity_weights_closed_form():
    """H = I, W_gate = W_up = W_down = identity, top_k = 1: out = bf16(SiLU(x) * x)."""
    H, E, T = 64, 4, 6
    eye = torch.eye(H).to(torch.bfloat16)
    W = eye.unsqueeze(0).repeat(E, 1, 1).contiguous()
    gen = torch.Generator().manual_seed(7)
    x = (3 * torch.randn(T, H, generator=gen)).to(torch.bfloat16)
    lg = torch.randn(T, E, generator=gen)
    r = oracle.forward(x, lg, W, W, W, top_k=1)
    xv = x.double().numpy()
    v = xv / (1.0 + np.exp(-xv)) * xv
    exp = f64_to_bf16_value(v)
    got = oracle.bf16_bits_to_f32(r["out"]).astype(np.float64)
    # equal, except possibly one bf16 ulp where v lies within fp32 error of a rounding tie
    ulp = bf16_ulp(v)
    near_tie = np.abs(np.abs(v - f64_to_bf16_value(v)) - ulp / 2) < 1e-5 * np.abs(v)
    ok = (got == exp) | (near_tie & (np.abs(got - exp) <= ulp))
    assert np.all(ok)


def test_zero_input_gives_zero():
    L = _tiny_layer(4, 32, 64, 9)
    x = torch.zeros(3, 32).to(torch.bfloat16)
    lg = torch.randn(3, 4, generator=torch.Generator().manual_seed(9))
    r = oracle.forward(x, lg, L["W_gate"], L["W_up"], L["W_down"], top_k=2)
    assert np.all(oracle.bf16_bits_to_f32(r["out"]) == 0.0)


def test_identical_experts_equal_one_dense_swiglu():
    """E identical experts with renormalised weights = one dense SwiGLU FFN."""
    E, H, I, T, k = 6, 32, 48, 5, 3
    one = _tiny_layer(1, H, I, 12)
    rep = {n: one[n].repeat(E, 1, 1).contiguous() for n in ("W_gate", "W_up", "W_down")}
    gen = torch.Generator().manual_seed(13)
    x = torch.randn(T, H, generator=gen).to(torch.bfloat16)
    lg = torch.randn(T, E, generator=gen)
    r = oracle.forward(x, lg, rep["W_gate"], rep["W_up"], rep["W_down"], top_k=k)
    dense = oracle.forward(x, torch.zeros(T, 1), one["W_gate"], one["W_up"], one["W_down"], top_k=1)
    d = dense["out_f32"].astype(np.float64)
    np.testing.assert_allclose(r["out_f32"], d, rtol=4e-6, atol=1e-12)


def test_token_permutation_permutes_output_exactly():
    E, H, I, T, k = 8, 32, 32, 9, 2
    L = _tiny_layer(E, H, I, 14)
    gen = torch.Generator().manual_seed(15)
    x = torch.randn(T, H, generator=gen).to(torch.bfloat16)
    lg = torch.randn(T, E, generator=gen)
    perm = torch.randperm(T, generator=gen)
    a = oracle.forward(x, lg, L["W_gate"], L["W_up"], L["W_down"], top_k=k)
    b = oracle.forward(x[perm], lg[perm], L["W_gate"], L["W_up"], L["W_down"], top_k=k)
    np.testing.assert_array_equal(b["out"], a["out"][perm.numpy()])


# ----------------------------------------------------------------------------
# INT8
def test_int8_power_of_two_scales_equal_bf16_exactly():
    """With scales 2^-n, q * s is exact in fp32 and in bf16, so the INT8 oracle must equal
    the BF16 oracle run on the dequantised weights bit for bit. Scales differ per (row,
    group), so a wrong group or row index in the dequantisation shows up."""
    E, H, I, T, k = 3, 256, 384, 4, 2
    gen = torch.Generator().manual_seed(21)
    q = {n: torch.randint(-127, 128, shape, generator=gen, dtype=torch.int8)
         for n, shape in (("g", (E, I, H)), ("u", (E, I, H)), ("d", (E, H, I)))}
    s = {n: torch.pow(2.0, -torch.randint(5, 11, (*q[n].shape[:-1], q[n].shape[-1] // 128), generator=gen).float())
         for n in q}
    deq = {n: (q[n].float() * torch.repeat_interleave(s[n], 128, dim=-1)).to(torch.bfloat16) for n in q}
    for n in q:  # the dequantised values are exactly representable in bf16
        assert torch.equal(deq[n].float(), q[n].float() * torch.repeat_interleave(s[n], 128, dim=-1))
    x = torch.randn(T, H, generator=gen).to(torch.bfloat16)
    lg = torch.randn(T, E, generator=gen)
    a = oracle.forward(x, lg, q["g"], q["u"], q["d"], s["g"], s["u"], s["d"], wtype="int8", top_k=k)
    b = oracle.forward(x, lg, deq["g"], deq["u"], deq["d"], top_k=k)
    np.testing.assert_array_equal(a["out_f32"], b["out_f32"])
    np.testing.assert_array_equal(a["out"], b["out"])


def test_int8_forward_matches_fp64_brute_force():
    E, H, I, T, k = 4, 256, 256, 3, 2
    L = _tiny_layer(E, H, I, 22, wtype="int8")
    gen = torch.Generator().manual_seed(23)
    x = torch.randn(T, H, generator=gen).to(torch.bfloat16)
    lg = torch.randn(T, E, generator=gen)
    r = oracle.forward(x, lg, L["W_gate"], L["W_up"], L["W_down"], L["s_gate"], L["s_up"], L["s_down"],
                       wtype="int8", top_k=k)
    b = brute_forward64(x, lg, L["W_gate"], L["W_up"], L["W_down"], k, L["s_gate"], L["s_up"], L["s_down"])
    ref = b["out"]
    # same structure of bound as the bf16 case, taken loosely: fp32 dequant adds one rounding
    assert np.max(np.abs(r["out_f32"] - ref)) <= 2e-3 * np.max(np.abs(ref))


def test_quantiser_properties():
    gen = torch.Generator().manual_seed(31)
    w = (0.02 * torch.randn(5, 7, 512, generator=gen)).to(torch.bfloat16)
    w[1, 2, 128:256] = 0  # one all-zero group
    q, s = mw.quantize_int8_groupwise(w)
    assert q.dtype == torch.int8 and s.shape == (5, 7, 4)
    assert s[1, 2, 1] == 1.0 and torch.all(q[1, 2, 128:256] == 0)
    deq = q.float() * torch.repeat_interleave(s, 128, dim=-1)
    err = (deq - w.float()).abs()
    # |w - q s| <= s/2 exactly; the fp32 division and product add a few ulp of 127 s
    assert torch.all(err <= torch.repeat_interleave(s, 128, dim=-1) * (0.5 + 1e-5))
    gmax = q.view(5, 7, 4, 128).abs().amax(-1)
    nz = w.float().view(5, 7, 4, 128).abs().amax(-1) > 0
    assert torch.all(gmax[nz] == 127)
    qn, sn = mw.quantize_int8_groupwise(-w)
    assert torch.equal(sn, s) and torch.equal(qn, -q)


def test_table3_shapes_golden():
    with open(os.path.join(GOLDEN, "table3_expert_shapes.json")) as f:
        models = json.load(f)["models"]
    for name, m in models.items():
        c = mw.CONFIGS[name]
        assert [c.H, c.I] == m["gate_up"] and [c.I, c.H] == m["down"], name
        assert c.top_k == m["top_k"] and c.E == m["experts"], name
    sk = mw.CONFIGS["mixtral8x22b_skew"]
    assert (sk.H, sk.I, sk.E, sk.top_k, sk.skew) == (6144, 16384, 8, 2, 2.0)
