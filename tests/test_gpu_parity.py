"""CUDA path vs the CPU oracle, element by element, through the C ABI (needs a GPU).

Integer routing outputs must be bit-exact. Float outputs must satisfy
|gpu - oracle| <= rel * max|oracle| + 1e-3 elementwise, rel = 1e-2 for bf16
weights and 2e-2 for int8 weights (identical q and scales on both sides).
"""
import numpy as np
import pytest
import torch

import moe_workloads as mw
import oracle
import routed_expert_ffn_softmax_gb300 as moe

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
REL = {"bf16": 1e-2, "int8": 2e-2}


@pytest.fixture(scope="module", autouse=True)
def _built():
    from routed_expert_ffn_softmax_gb300 import build
    build.build()
    moe.load()
    yield


def to_np_f32(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy()


def assert_moe_close(gpu: np.ndarray, ref: np.ndarray, wtype: str, what: str = ""):
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    assert np.all(np.isfinite(gpu)), f"{what}: non-finite output"
    bound = REL[wtype] * np.max(np.abs(ref)) + 1e-3
    err = np.abs(gpu - ref)
    assert np.all(err <= bound), f"{what}: max err {err.max():.4g} > bound {bound:.4g}"


def gpu_route(logits: torch.Tensor, k: int):
    T, E = logits.shape
    P = T * k
    i32 = dict(dtype=torch.int32, device=logits.device)
    o = dict(ids=torch.full((T, k), -1, **i32), w=torch.full((T, k), -1.0, device=logits.device),
             counts=torch.full((E,), -1, **i32), offsets=torch.full((E + 1,), -1, **i32),
             sorted_token=torch.full((P,), -1, **i32), inv_pos=torch.full((T, k), -1, **i32),
             active=torch.full((E,), -1, **i32), num_active=torch.full((1,), -1, **i32))
    moe.moe_route_topk(logits, k, o["ids"], o["w"], o["counts"], o["offsets"], o["sorted_token"], o["inv_pos"],
                       o["active"], o["num_active"])
    torch.cuda.synchronize()
    return {n: v.cpu().numpy() for n, v in o.items()}


def check_route(r_gpu, r_ora):
    for n in ("ids", "counts", "offsets", "sorted_token", "inv_pos"):
        np.testing.assert_array_equal(r_gpu[n], r_ora[n], err_msg=n)
    na = int(r_gpu["num_active"][0])
    assert na == r_ora["num_active"]
    np.testing.assert_array_equal(r_gpu["active"][:na], r_ora["active"])
    np.testing.assert_allclose(r_gpu["w"], r_ora["w"], rtol=1e-6, atol=1e-7)


# ------------------------------------------------------------------ routing
@pytest.mark.parametrize("T,E,k", [(1, 8, 2), (7, 8, 2), (64, 8, 2), (512, 256, 8), (256, 128, 8), (3, 5, 5),
                                   (1500, 64, 4), (33, 256, 1), (2048, 256, 8)])
def test_route_bit_exact(T, E, k):
    g = torch.Generator(device=DEV).manual_seed(T * 7 + E)
    lg = torch.randn(T, E, generator=g, device=DEV)
    check_route(gpu_route(lg, k), oracle.route(lg.cpu(), k))


def test_route_ties_and_skew():
    g = torch.Generator(device=DEV).manual_seed(5)
    lg = torch.randint(-2, 3, (300, 32), generator=g, device=DEV).float()  # many exact ties
    check_route(gpu_route(lg, 4), oracle.route(lg.cpu(), 4))
    lg = torch.randn(64, 8, generator=g, device=DEV)
    lg[:, :2] += 2.0
    check_route(gpu_route(lg, 2), oracle.route(lg.cpu(), 2))


def test_route_golden_cases():
    import json, os
    with open(os.path.join(os.path.dirname(__file__), "golden", "routing_worked.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        lg = torch.tensor(c["logits"], dtype=torch.float32, device=DEV)
        r = gpu_route(lg, c["top_k"])
        np.testing.assert_array_equal(r["ids"], np.array(c["ids"]), err_msg=c["name"])
        if "w" in c:
            np.testing.assert_allclose(r["w"], np.array(c["w"]), rtol=1e-6, err_msg=c["name"])
        for key in ("counts", "offsets", "sorted_token", "inv_pos"):
            if key in c:
                np.testing.assert_array_equal(r[key], np.array(c[key]), err_msg=f"{c['name']}:{key}")


# ------------------------------------------------------------------ gather / combine
def test_gather_is_row_copy():
    T, H, E, k = 37, 264, 16, 3
    g = torch.Generator(device=DEV).manual_seed(1)
    x = torch.randn(T, H, generator=g, device=DEV).to(torch.bfloat16)
    lg = torch.randn(T, E, generator=g, device=DEV)
    r = oracle.route(lg.cpu(), k)
    st = torch.from_numpy(r["sorted_token"]).to(DEV)
    xg = torch.empty(T * k, H, dtype=torch.bfloat16, device=DEV)
    moe.moe_gather(x, k, st, xg)
    torch.cuda.synchronize()
    assert torch.equal(xg.cpu(), x.cpu()[torch.from_numpy(r["sorted_token"]).long()])


def test_combine_bit_exact():
    T, H, E, k = 19, 136, 8, 3
    g = torch.Generator(device=DEV).manual_seed(2)
    lg = torch.randn(T, E, generator=g, device=DEV)
    r = oracle.route(lg.cpu(), k)
    Y = torch.randn(T * k, H, generator=g, device=DEV)
    out = torch.empty(T, H, dtype=torch.bfloat16, device=DEV)
    moe.moe_combine(Y, torch.from_numpy(r["inv_pos"]).to(DEV), torch.from_numpy(r["w"]).to(DEV), k, out)
    torch.cuda.synchronize()
    Yc = Y.cpu().numpy()
    got = out.cpu().view(torch.int16).numpy().view(np.uint16)
    for t in range(T):
        ref, _ = oracle.combine_token(Yc[r["inv_pos"][t]], r["w"][t])
        np.testing.assert_array_equal(got[t], ref)


# ------------------------------------------------------------------ expert FFN / forward, small
def small_case(T, H, I, E, k, wtype, seed, skew=()):
    cfg = mw.MoEConfig("case", H, I, E, k, wtype, (T,), skew_experts=tuple(skew), skew=3.0 if skew else 0.0)
    L = mw.make_layer(cfg, seed=seed, device="cpu")
    x, lg = mw.make_tokens(cfg, T, seed=seed, device="cpu")
    return cfg, L, x, lg


def run_forward_ws(L, x, lg, k):
    dev = {n: (v.to(DEV) if v is not None else None) for n, v in L.items()}
    T, H = x.shape
    E, I, _ = L["W_gate"].shape
    wt = moe.MOE_W_INT8_G128 if L["W_gate"].dtype == torch.int8 else moe.MOE_W_BF16
    ws = moe.alloc_workspace(T, H, I, E, k, wt, DEV)
    out = torch.full((T, H), float("nan"), dtype=torch.bfloat16, device=DEV)
    moe.moe_ffn_forward(x.to(DEV), lg.to(DEV), dev["W_gate"], dev["W_up"], dev["W_down"], dev["s_gate"],
                        dev["s_up"], dev["s_down"], k, out, ws)
    torch.cuda.synchronize()
    assert moe.workspace_status(ws) == 0
    return out, ws


SMALL = [
    # T, H, I, E, k, wtype, skew     (several tiles, ragged tails, multi-pass experts)
    (8, 256, 512, 8, 2, "bf16", ()),        # the tiny workload
    (1, 256, 512, 8, 2, "bf16", ()),
    (5, 200, 136, 6, 2, "bf16", ()),        # H, I not multiples of 64 / 128
    (96, 128, 192, 3, 2, "bf16", ()),       # ~64 tokens per expert
    (150, 64, 256, 4, 2, "bf16", (0, 1)),   # skewed: experts 0,1 get > 64 tokens (several passes)
    (40, 512, 384, 16, 16, "bf16", ()),     # top_k = E
    (12, 256, 256, 32, 1, "bf16", ()),      # top_k = 1
    (4, 256, 384, 8, 2, "int8", ()),
    (70, 384, 256, 8, 4, "int8", (2,)),
    (36, 256, 384, 8, 2, "int8", (3,)),     # 16-token passes (P <= 9 E), expert 3 past one pass
    (56, 256, 256, 8, 2, "int8", (6,)),     # 32-token passes (P > 9 E): 2 for expert 6, 1 for the rest
    (60, 256, 256, 8, 2, "bf16", (1,)),     # one tile shape for the launch, set by expert 1's pass
    # about one token per expert (P = T * k <= E)
    (3, 264, 200, 8, 2, "bf16", ()),        # H, I not multiples of 64
    (6, 256, 512, 16, 2, "bf16", (0,)),     # expert 0 gets ~6 tokens, the others 0-1
    (2, 128, 128, 4, 2, "int8", ()),
    (8, 640, 384, 64, 8, "int8", (5,)),     # expert 5 gets all 8 tokens, 56 others one each
]


@pytest.mark.parametrize("T,H,I,E,k,wtype,skew", SMALL)
def test_forward_matches_oracle_small(T, H, I, E, k, wtype, skew):
    cfg, L, x, lg = small_case(T, H, I, E, k, wtype, seed=T + H + E, skew=skew)
    out, _ = run_forward_ws(L, x, lg, k)
    ref = oracle.forward(x, lg, L["W_gate"], L["W_up"], L["W_down"], L["s_gate"], L["s_up"], L["s_down"],
                         wtype=wtype, top_k=k)
    assert_moe_close(to_np_f32(out), oracle.bf16_bits_to_f32(ref["out"]), wtype, f"T={T} H={H} I={I} E={E} k={k}")


@pytest.mark.parametrize("T,H,I,E,k,wtype,skew", [SMALL[2], SMALL[4], SMALL[8]])
def test_expert_ffn_entry_point_matches_oracle(T, H, I, E, k, wtype, skew):
    """moe_route_topk -> moe_gather -> moe_expert_ffn -> moe_combine, each called separately;
    Y compared with the oracle's per-assignment expert outputs."""
    cfg, L, x, lg = small_case(T, H, I, E, k, wtype, seed=11 * T + H, skew=skew)
    dev = {n: (v.to(DEV) if v is not None else None) for n, v in L.items()}
    r = gpu_route(lg.to(DEV), k)
    ro = oracle.route(lg, k)
    check_route(r, ro)
    P = T * k
    xg = torch.empty(P, H, dtype=torch.bfloat16, device=DEV)
    st = torch.from_numpy(r["sorted_token"]).to(DEV)
    moe.moe_gather(x.to(DEV), k, st, xg)
    Y = torch.full((P, H), float("nan"), device=DEV)
    wt = moe.MOE_W_INT8_G128 if wtype == "int8" else moe.MOE_W_BF16
    ws = moe.alloc_workspace(T, H, I, E, k, wt, DEV)
    moe.moe_expert_ffn(xg, torch.from_numpy(r["offsets"]).to(DEV), torch.from_numpy(r["active"]).to(DEV),
                       torch.from_numpy(r["num_active"]).to(DEV), dev["W_gate"], dev["W_up"], dev["W_down"],
                       dev["s_gate"], dev["s_up"], dev["s_down"], Y, ws)
    out = torch.empty(T, H, dtype=torch.bfloat16, device=DEV)
    moe.moe_combine(Y, torch.from_numpy(r["inv_pos"]).to(DEV), torch.from_numpy(r["w"]).to(DEV), k, out)
    torch.cuda.synchronize()
    assert moe.workspace_status(ws) == 0
    Yc = Y.cpu().numpy()
    xb = x.contiguous()
    for t in range(T):
        for j in range(k):
            e = int(ro["ids"][t, j])
            sc = (lambda n: L[n][e] if L[n] is not None else None)
            h, _, _ = oracle.gateup_token(xb[t], L["W_gate"][e], L["W_up"][e], sc("s_gate"), sc("s_up"), wtype)
            y = oracle.down_token(h, L["W_down"][e], sc("s_down"), wtype)
            assert_moe_close(Yc[ro["inv_pos"][t, j]], y, wtype, f"Y t={t} j={j}")
    ref = oracle.forward(x, lg, L["W_gate"], L["W_up"], L["W_down"], L["s_gate"], L["s_up"], L["s_down"],
                         wtype=wtype, top_k=k)
    assert_moe_close(to_np_f32(out), oracle.bf16_bits_to_f32(ref["out"]), wtype, "out")


@pytest.mark.parametrize("T", [9, 4])
@pytest.mark.parametrize("x_scale", [2.0 ** 17, 2.0 ** -30, 1.0])
def test_int8_activation_range(x_scale, T):
    """INT8 runs the tensor cores in fp16; token rows far outside fp16's range (large or tiny)
    must still match the oracle to a purely relative bound."""
    H, I, E, k = 256, 384, 8, 2
    cfg, L, x, lg = small_case(T, H, I, E, k, "int8", seed=77)
    xs = (x.float() * x_scale).to(torch.bfloat16)
    out, _ = run_forward_ws(L, xs, lg, k)
    ref = oracle.forward(xs, lg, L["W_gate"], L["W_up"], L["W_down"], L["s_gate"], L["s_up"], L["s_down"],
                         wtype="int8", top_k=k)
    r = oracle.bf16_bits_to_f32(ref["out"]).astype(np.float64)
    g = to_np_f32(out).astype(np.float64)
    assert np.all(np.isfinite(g)) and np.abs(r).max() > 0
    assert np.abs(g - r).max() <= 2e-2 * np.abs(r).max()


def test_forward_is_deterministic_and_repeatable():
    cfg, L, x, lg = small_case(64, 512, 1024, 8, 2, "bf16", seed=3)
    a, ws = run_forward_ws(L, x, lg, 2)
    b, _ = run_forward_ws(L, x, lg, 2)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_forward_zero_tokens_is_noop():
    cfg, L, x, lg = small_case(4, 256, 512, 8, 2, "bf16", seed=4)
    dev = {n: (v.to(DEV) if v is not None else None) for n, v in L.items()}
    out = torch.full((0, 256), 7.0, dtype=torch.bfloat16, device=DEV)
    ws = moe.alloc_workspace(1, 256, 512, 8, 2, moe.MOE_W_BF16, DEV)
    moe.moe_ffn_forward(x[:0].to(DEV), lg[:0].to(DEV), dev["W_gate"], dev["W_up"], dev["W_down"], None, None, None,
                        2, out, ws)
    torch.cuda.synchronize()


# ------------------------------------------------------------------ full-size workloads, every token
def oracle_rows(cfg, Lc, x, lg, tokens=None):
    """Oracle output rows (fp32 values of the bf16 outputs) for `tokens` (default: all), computed
    one token-expert assignment at a time from the CPU copy of the layer, and the oracle's routing."""
    ro = oracle.route(lg, cfg.top_k)
    tokens = range(x.shape[0]) if tokens is None else tokens
    rows = {}
    for t in tokens:
        ys = []
        for j in range(cfg.top_k):
            e = int(ro["ids"][t, j])
            sc = (lambda n: Lc[n][e] if Lc[n] is not None else None)
            h, _, _ = oracle.gateup_token(x[t], Lc["W_gate"][e], Lc["W_up"][e], sc("s_gate"), sc("s_up"), cfg.wtype)
            ys.append(oracle.down_token(h, Lc["W_down"][e], sc("s_down"), cfg.wtype))
        out, _ = oracle.combine_token(np.stack(ys), ro["w"][t])
        rows[t] = oracle.bf16_bits_to_f32(out)
    return ro, rows


# Every (config, T) point of the four full-size expert shapes (HiNa-MoE §8.1 Table 3 at 1-16
# tokens per expert), plus INT8 at 2 and 4 tokens, where by batch shape the one-launch decode step
# runs; in config order so that one config's layer serves all its T.
FULL = [(name, T) for name in ("mixtral8x7b", "mixtral8x22b", "mixtral8x22b_skew", "dsv3", "qwen3_int8")
        for T in sorted(set(mw.CONFIGS[name].T) | ({2, 4} if name == "qwen3_int8" else set()))]

_LAYERS = {}


def full_layer(name):
    """The config's layer on the device and its CPU copy; one config is held at a time (the skewed
    8x22B variant shares the 8x22B weights: only its router logits differ)."""
    key = "mixtral8x22b" if name == "mixtral8x22b_skew" else name
    if key not in _LAYERS:
        _LAYERS.clear()
        torch.cuda.empty_cache()
        Lg = mw.make_layer(mw.CONFIGS[key], device=DEV)
        Lc = {n: (v.cpu() if v is not None else None) for n, v in Lg.items()}
        _LAYERS[key] = (Lg, Lc)
    return _LAYERS[key]


@pytest.fixture(scope="module")
def _release_layers():
    yield
    _LAYERS.clear()
    torch.cuda.empty_cache()


@pytest.mark.parametrize("name,T", FULL)
def test_full_size_every_token(name, T, _release_layers):
    """moe_ffn_forward on the full-size layer; every token's output row against the oracle, and the
    whole batch's routing bit-exact."""
    cfg = mw.CONFIGS[name]
    Lg, Lc = full_layer(name)
    x, lg = mw.make_tokens(cfg, T, device=DEV)
    wt = moe.MOE_W_INT8_G128 if cfg.wtype == "int8" else moe.MOE_W_BF16
    ws = moe.alloc_workspace(T, cfg.H, cfg.I, cfg.E, cfg.top_k, wt, DEV)
    out = torch.full((T, cfg.H), float("nan"), dtype=torch.bfloat16, device=DEV)
    moe.moe_ffn_forward(x, lg, Lg["W_gate"], Lg["W_up"], Lg["W_down"], Lg["s_gate"], Lg["s_up"], Lg["s_down"],
                        cfg.top_k, out, ws)
    torch.cuda.synchronize()
    assert moe.workspace_status(ws) == 0
    got = to_np_f32(out)
    assert np.all(np.isfinite(got))
    ro, rows = oracle_rows(cfg, Lc, x.cpu(), lg.cpu())
    for t in range(T):
        assert_moe_close(got[t], rows[t], cfg.wtype, f"{name} T={T} token {t}")
    check_route(gpu_route(lg, cfg.top_k), ro)
