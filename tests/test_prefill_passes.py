"""The BF16 expert kernels at prefill sizes (HiNa-MoE §8.2 "Prefill Phase": many tokens per expert),
against the CPU oracle through the C ABI (needs a GPU).

At 128- and 256-token passes an expert with more tokens than one pass is split evenly over up to
4 CTAs (ranks) that take the same weight blocks side by side; more than 4 passes' worth take further
rounds. These cases cover: one and several ranks, a second round, ranks left without tokens,
reduction lengths and row counts that are not multiples of a tile (TMA zero fill), every pass size
forced for gate+up and for down independently, and the full-size Mixtral-8x7B expert shape at 256
and 512 tokens per expert on sampled tokens.
"""
import numpy as np
import pytest
import torch

import moe_workloads as mw
import oracle
import routed_expert_ffn_softmax_gb300 as moe
from test_gpu_parity import DEV, assert_moe_close, check_route, gpu_route, oracle_rows, small_case, to_np_f32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from routed_expert_ffn_softmax_gb300 import build
    build.build()
    moe.load()
    yield
    moe.moe_set_expert_pass_tokens(0, 0)


def forward(L, x, lg, k, passes=(0, 0)):
    """moe_ffn_forward with the given pass sizes (the workspace sized under them)."""
    T, H = x.shape
    E, I, _ = L["W_gate"].shape
    moe.moe_set_expert_pass_tokens(*passes)
    try:
        ws = moe.alloc_workspace(T, H, I, E, k, moe.MOE_W_BF16, DEV)
        out = torch.full((T, H), float("nan"), dtype=torch.bfloat16, device=DEV)
        moe.moe_ffn_forward(x, lg, L["W_gate"], L["W_up"], L["W_down"], None, None, None, k, out, ws)
        torch.cuda.synchronize()
    finally:
        moe.moe_set_expert_pass_tokens(0, 0)
    assert moe.workspace_status(ws) == 0
    ctrl = ws[:4096].view(torch.int32).cpu().numpy()
    assert not ctrl[64:64 + 256].any(), "stream-K counters must be left at zero"
    return out


CASES = [
    # T, H, I, E, k, skew          tokens per expert (mean), what it covers
    (600, 256, 512, 4, 2, ()),      # 300: 256-token passes, 2 ranks
    (200, 128, 256, 4, 2, ()),      # 100: 256-token passes, 1 rank
    (1500, 128, 128, 4, 1, (0,)),   # expert 0 past 4 x 256 tokens: 4 ranks, a second round
    (300, 200, 136, 6, 2, ()),      # 100: reduction 200 and rows 136 are ragged (zero-filled tiles)
    (160, 256, 384, 8, 2, (1,)),    # 40: 64-token passes; expert 1 several
    (400, 192, 320, 16, 4, ()),     # 100: 16 experts
]


@pytest.mark.parametrize("T,H,I,E,k,skew", CASES)
def test_prefill_matches_oracle(T, H, I, E, k, skew):
    cfg, L, x, lg = small_case(T, H, I, E, k, "bf16", seed=T + 7 * H + E, skew=skew)
    dev = {n: (v.to(DEV) if v is not None else None) for n, v in L.items()}
    out = forward(dev, x.to(DEV), lg.to(DEV), k)
    ref = oracle.forward(x, lg, L["W_gate"], L["W_up"], L["W_down"], wtype="bf16", top_k=k)
    assert_moe_close(to_np_f32(out), oracle.bf16_bits_to_f32(ref["out"]), "bf16", f"T={T} H={H} I={I} E={E}")


@pytest.mark.parametrize("passes", [(64, 64), (128, 128), (192, 192), (256, 256), (128, 256), (256, 64), (64, 128),
                                    (192, 64)])
def test_every_pass_size_matches_oracle(passes):
    """Each gate+up / down pass size on one skewed batch (experts 0 and 1 hot): ranks, rounds, and ranks
    left without tokens all occur for some pass size."""
    T, H, I, E, k = 700, 128, 384, 6, 2
    cfg, L, x, lg = small_case(T, H, I, E, k, "bf16", seed=5, skew=(0, 1))
    dev = {n: (v.to(DEV) if v is not None else None) for n, v in L.items()}
    out = forward(dev, x.to(DEV), lg.to(DEV), k, passes)
    ref = oracle.forward(x, lg, L["W_gate"], L["W_up"], L["W_down"], wtype="bf16", top_k=k)
    assert_moe_close(to_np_f32(out), oracle.bf16_bits_to_f32(ref["out"]), "bf16", f"passes {passes}")


def test_workspace_sized_for_smaller_passes_is_rejected():
    """A workspace sized while 64-token passes were in force is too small once 256 is forced (the partial
    slots grow): both entry points return MOE_ERR_WORKSPACE and launch nothing; a workspace sized
    afterwards runs and matches the oracle."""
    T, H, I, E, k = 40, 256, 256, 8, 2
    cfg, L, x, lg = small_case(T, H, I, E, k, "bf16", seed=9, skew=(2,))
    dev = {n: (v.to(DEV) if v is not None else None) for n, v in L.items()}
    xd, lgd = x.to(DEV), lg.to(DEV)
    ws = moe.alloc_workspace(T, H, I, E, k, moe.MOE_W_BF16, DEV)
    out = torch.full((T, H), float("nan"), dtype=torch.bfloat16, device=DEV)
    P = T * k
    r = gpu_route(lgd, k)
    xg = torch.empty(P, H, dtype=torch.bfloat16, device=DEV)
    moe.moe_gather(xd, k, torch.from_numpy(r["sorted_token"]).to(DEV), xg)
    Y = torch.full((P, H), float("nan"), device=DEV)
    moe.moe_set_expert_pass_tokens(256, 256)
    try:
        with pytest.raises(moe.MoeError, match="WORKSPACE"):
            moe.moe_ffn_forward(xd, lgd, dev["W_gate"], dev["W_up"], dev["W_down"], None, None, None, k, out, ws)
        with pytest.raises(moe.MoeError, match="WORKSPACE"):
            moe.moe_expert_ffn(xg, torch.from_numpy(r["offsets"]).to(DEV), torch.from_numpy(r["active"]).to(DEV),
                               torch.from_numpy(r["num_active"]).to(DEV), dev["W_gate"], dev["W_up"],
                               dev["W_down"], None, None, None, Y, ws)
        torch.cuda.synchronize()
    finally:
        moe.moe_set_expert_pass_tokens(0, 0)
    assert torch.isnan(out.float()).all() and torch.isnan(Y).all()  # nothing was written
    got = forward(dev, xd, lgd, k, (256, 256))
    ref = oracle.forward(x, lg, L["W_gate"], L["W_up"], L["W_down"], wtype="bf16", top_k=k)
    assert_moe_close(to_np_f32(got), oracle.bf16_bits_to_f32(ref["out"]), "bf16", "256-token passes")


def sample_tokens(ro, E, per_expert_positions, seed):
    """Tokens whose assignments sit at the given positions within their expert's segment (first and last
    row, pass and rank boundaries), plus a few at random."""
    off, st = ro["offsets"], ro["sorted_token"]
    picks = set()
    for e in range(E):
        n = int(off[e + 1] - off[e])
        for p in per_expert_positions + [n - 1]:
            if 0 <= p < n:
                picks.add(int(st[off[e] + p]))
    rng = np.random.default_rng(seed)
    picks.update(int(t) for t in rng.choice(len(ro["ids"]), 8, replace=False))
    return sorted(picks)


@pytest.mark.parametrize("T", [256, 1024, 2048])
def test_full_size_prefill_sampled(T):
    """Mixtral-8x7B expert shape (H 4096, I 14336, top-2 of 8) at 64 (128-token passes), 256 and 512
    tokens per expert (256-token passes): every expert's first and last rows and rows at multiples of
    128 around the rank boundaries, against the oracle token by token; the routing bit-exact."""
    cfg = mw.CONFIGS["mixtral8x7b_prefill"]
    Lg = mw.make_layer(cfg, device=DEV)
    x, lg = mw.make_tokens(cfg, T, device=DEV)
    out = forward(Lg, x, lg, cfg.top_k)
    got = to_np_f32(out)
    assert np.all(np.isfinite(got))
    Lc = {n: (v.cpu() if v is not None else None) for n, v in Lg.items()}
    del Lg
    torch.cuda.empty_cache()
    ro = oracle.route(lg.cpu(), cfg.top_k)
    check_route(gpu_route(lg, cfg.top_k), ro)
    positions = [0, 1, 127, 128, 255, 256, 257, 383, 384, 511, 512]
    tokens = sample_tokens(ro, cfg.E, positions if T == 2048 else positions[:7 if T == 1024 else 4], seed=T)
    _, rows = oracle_rows(cfg, Lc, x.cpu(), lg.cpu(), tokens)
    for t in tokens:
        assert_moe_close(got[t], rows[t], "bf16", f"prefill T={T} token {t}")


@pytest.mark.parametrize("T", [4096])
def test_full_size_dsv3_prefill_sampled(T):
    """DeepSeek-V3 expert shape (H 7168, I 2048, top-8 of 256) at 128 tokens per expert: pair kernels with
    192-token passes over 256 experts. Every expert's first and last rows and a few at random, against
    the oracle token by token (the first 32 experts' rows only, to bound the oracle's time); the routing
    bit-exact."""
    cfg = mw.CONFIGS["dsv3_prefill"]
    Lg = mw.make_layer(cfg, device=DEV)
    x, lg = mw.make_tokens(cfg, T, device=DEV)
    out = forward(Lg, x, lg, cfg.top_k)
    got = to_np_f32(out)
    assert np.all(np.isfinite(got))
    ro = oracle.route(lg.cpu(), cfg.top_k)
    check_route(gpu_route(lg, cfg.top_k), ro)
    off, st = ro["offsets"], ro["sorted_token"]
    picks = set()
    for e in range(0, cfg.E, 8):  # every eighth expert: first, 64th and last rows
        n = int(off[e + 1] - off[e])
        for p in (0, 63, 64, n - 1):
            if 0 <= p < n:
                picks.add(int(st[off[e] + p]))
    tokens = sorted(picks)[:48]
    Lc = {n: (v.cpu() if v is not None else None) for n, v in Lg.items()}
    del Lg
    torch.cuda.empty_cache()
    _, rows = oracle_rows(cfg, Lc, x.cpu(), lg.cpu(), tokens)
    for t in tokens:
        assert_moe_close(got[t], rows[t], "bf16", f"dsv3 prefill T={T} token {t}")
