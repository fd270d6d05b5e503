"""The one-launch decode step (routing, gate+up, down and combine in one cooperative kernel) against
the CPU oracle, element by element, through the C ABI (needs a GPU).

moe_ffn_forward takes this path for small decode batches; here the policy forces it (2) so that every
shape below runs it (passes of 1 token at T = 1, of 4 when P <= E, of 8 above), including skewed batches
whose hot experts need several passes, and
checks it against the oracle and against the staged path (policy 1). The workspace's counters must be
back at zero after every call, so that consecutive calls on one workspace need no clearing.
"""
import numpy as np
import pytest
import torch

import moe_workloads as mw
import oracle
import routed_expert_ffn_softmax_gb300 as moe
from test_gpu_parity import DEV, assert_moe_close, check_route, small_case, to_np_f32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from routed_expert_ffn_softmax_gb300 import build
    build.build()
    moe.load()
    yield
    moe.moe_set_decode_step_policy(0)


def forward(L, x, lg, k, policy, ws=None):
    T, H = x.shape
    E, I, _ = L["W_gate"].shape
    wt = moe.MOE_W_INT8_G128 if L["W_gate"].dtype == torch.int8 else moe.MOE_W_BF16
    moe.moe_set_decode_step_policy(policy)
    try:
        if ws is None:
            ws = moe.alloc_workspace(T, H, I, E, k, wt, DEV)
        out = torch.full((T, H), float("nan"), dtype=torch.bfloat16, device=DEV)
        moe.moe_ffn_forward(x, lg, L["W_gate"], L["W_up"], L["W_down"], L["s_gate"], L["s_up"], L["s_down"], k, out,
                            ws)
        torch.cuda.synchronize()
    finally:
        moe.moe_set_decode_step_policy(0)
    assert moe.workspace_status(ws) == 0
    return out, ws


def ctrl_words(ws):
    """(grid-barrier arrivals, stream-K counters, row-block counters) of a workspace."""
    w = ws[:4096].view(torch.int32).cpu().numpy()
    return int(w[2]), w[64:64 + 256], w[512:1024]


def routing_in_workspace(ws, T, H, I, E, k, int8):
    """The routing tables the call left in its workspace (the layout of csrc/api.cu)."""
    P = T * k
    off = 4096 + 4 * 256 * 2 * 16384  # ctrl, partials
    up = lambda n: (n + 255) // 256 * 256
    off += up(2 * P * I)
    if int8:
        off += up(2 * P * I) + up(2 * P * H) + 2 * up(4 * P)
    b = ws.cpu().numpy()

    def take(n, dtype):
        nonlocal off
        a = b[off:off + 4 * n].view(dtype).copy()
        off += up(4 * n)
        return a
    r = {}
    r["ids"] = take(P, np.int32).reshape(T, k)
    r["w"] = take(P, np.float32).reshape(T, k)
    r["counts"] = take(E, np.int32)
    r["offsets"] = take(E + 1, np.int32)
    r["sorted_token"] = take(P, np.int32)
    r["inv_pos"] = take(P, np.int32).reshape(T, k)
    r["active"] = take(E, np.int32)
    r["num_active"] = take(1, np.int32)
    return r


CASES = [
    # T, H, I, E, k, wtype, skew          (about one token per expert; passes of 8; ragged stream-K splits)
    (1, 256, 512, 8, 2, "bf16", ()),
    (8, 256, 512, 8, 2, "bf16", ()),              # the tiny workload
    (3, 384, 640, 16, 4, "bf16", ()),
    (32, 512, 256, 64, 4, "bf16", ()),            # 32 tokens, 128 assignments over 64 experts
    (20, 256, 384, 8, 2, "bf16", (0,)),           # expert 0 gets ~20 tokens: three passes
    (6, 128, 128, 4, 4, "bf16", ()),              # top_k = E
    (5, 1024, 256, 256, 8, "bf16", ()),           # E = 256 (eight logits per lane)
    (1, 512, 512, 128, 8, "int8", ()),
    (8, 1024, 512, 128, 8, "int8", ()),
    (16, 512, 1024, 32, 2, "int8", (3,)),         # expert 3 gets every token: two passes
    (32, 512, 512, 64, 8, "int8", ()),            # P = 256
    (2, 1536, 512, 8, 2, "int8", ()),
    # passes of 4 tokens (at most one assignment per expert on average): a hot expert takes several
    (8, 512, 512, 64, 2, "bf16", (0,)),           # expert 0 gets all 8 tokens: two passes
    (12, 512, 512, 64, 4, "int8", (1,)),          # expert 1 gets all 12: three passes
]


@pytest.mark.parametrize("T,H,I,E,k,wtype,skew", CASES)
def test_decode_step_matches_oracle(T, H, I, E, k, wtype, skew):
    cfg, L, x, lg = small_case(T, H, I, E, k, wtype, seed=3 * T + H + E, skew=skew)
    assert moe.moe_ffn_forward_launches(T, H, I, E, k, cfg.wtype == "int8") in (1, 5, 6)
    dev = {n: (v.to(DEV) if v is not None else None) for n, v in L.items()}
    xd, lgd = x.to(DEV), lg.to(DEV)
    out, ws = forward(dev, xd, lgd, k, policy=2)
    ref = oracle.forward(x, lg, L["W_gate"], L["W_up"], L["W_down"], L["s_gate"], L["s_up"], L["s_down"],
                         wtype=wtype, top_k=k)
    assert_moe_close(to_np_f32(out), oracle.bf16_bits_to_f32(ref["out"]), wtype, f"decode step T={T} H={H} E={E}")
    # the routing tables it leaves in the workspace are the definition's, bit for bit
    r = routing_in_workspace(ws, T, H, I, E, k, wtype == "int8")
    check_route(r, oracle.route(lg, k))
    # counters back at zero: the next call on this workspace needs no clearing
    arrivals, counters, rows = ctrl_words(ws)
    assert arrivals == 0 and not counters.any() and not rows.any()
    # the staged path on the same inputs agrees within the same bound
    staged, _ = forward(dev, xd, lgd, k, policy=1)
    assert_moe_close(to_np_f32(out), to_np_f32(staged), wtype, "decode step vs staged path")


@pytest.mark.parametrize("wtype", ["bf16", "int8"])
def test_decode_step_reuses_its_workspace(wtype):
    """Three consecutive calls on one workspace (different batches), each oracle-checked, and a repeat of
    the first batch bit-identical to its first run."""
    T, H, I, E, k = 4, 512, 512, 16, 4
    cfg, L, _, _ = small_case(T, H, I, E, k, wtype, seed=91)
    dev = {n: (v.to(DEV) if v is not None else None) for n, v in L.items()}
    ws = None
    outs = []
    for s in (1, 2, 3, 1):
        x, lg = mw.make_tokens(cfg, T, seed=s)
        out, ws = forward(dev, x.to(DEV), lg.to(DEV), k, policy=2, ws=ws)
        ref = oracle.forward(x, lg, L["W_gate"], L["W_up"], L["W_down"], L["s_gate"], L["s_up"], L["s_down"],
                             wtype=wtype, top_k=k)
        assert_moe_close(to_np_f32(out), oracle.bf16_bits_to_f32(ref["out"]), wtype, f"batch {s}")
        outs.append(out)
    assert torch.equal(outs[0].view(torch.int16), outs[3].view(torch.int16))


@pytest.mark.parametrize("x_scale", [2.0 ** 17, 2.0 ** -30])
def test_decode_step_int8_activation_range(x_scale):
    """fp16 copies of the tokens (row scale) and of h (group scale) keep far-from-unit rows exact."""
    T, H, I, E, k = 3, 512, 512, 8, 2
    cfg, L, x, lg = small_case(T, H, I, E, k, "int8", seed=44)
    xs = (x.float() * x_scale).to(torch.bfloat16)
    dev = {n: (v.to(DEV) if v is not None else None) for n, v in L.items()}
    out, _ = forward(dev, xs.to(DEV), lg.to(DEV), k, policy=2)
    ref = oracle.forward(xs, lg, L["W_gate"], L["W_up"], L["W_down"], L["s_gate"], L["s_up"], L["s_down"],
                         wtype="int8", top_k=k)
    r = oracle.bf16_bits_to_f32(ref["out"]).astype(np.float64)
    g = to_np_f32(out).astype(np.float64)
    assert np.all(np.isfinite(g)) and np.abs(r).max() > 0
    assert np.abs(g - r).max() <= 2e-2 * np.abs(r).max()


def test_grid_barrier_expiry_reports_status_and_the_gpu_recovers():
    """The bounded wait on another CTA, made to run out: with the test hook on, the decode step's grid
    barrier expects one CTA more than the launch has, so it never opens; every CTA gives up after 20 ms,
    the call returns, the workspace status word reads 5 (the grid-barrier timeout). Then, with the hook
    off and the workspace zeroed again, a normal call on the same GPU is oracle-green with status 0."""
    T, H, I, E, k = 2, 512, 512, 8, 2
    cfg, L, x, lg = small_case(T, H, I, E, k, "bf16", seed=123)
    dev = {n: (v.to(DEV) if v is not None else None) for n, v in L.items()}
    xd, lgd = x.to(DEV), lg.to(DEV)
    ws = moe.alloc_workspace(T, H, I, E, k, moe.MOE_W_BF16, DEV)
    out = torch.empty(T, H, dtype=torch.bfloat16, device=DEV)
    moe.moe_set_decode_step_policy(2)
    try:
        moe.moe_test_expire_grid_barrier(True, 20_000_000)
        moe.moe_ffn_forward(xd, lgd, dev["W_gate"], dev["W_up"], dev["W_down"], None, None, None, k, out, ws)
        torch.cuda.synchronize()
    finally:
        moe.moe_test_expire_grid_barrier(False)
        moe.moe_set_decode_step_policy(0)
    assert moe.workspace_status(ws) == 5
    ws.zero_()
    good, ws2 = forward(dev, xd, lgd, k, policy=2, ws=ws)
    ref = oracle.forward(x, lg, L["W_gate"], L["W_up"], L["W_down"], top_k=k)
    assert_moe_close(to_np_f32(good), oracle.bf16_bits_to_f32(ref["out"]), "bf16", "after the expired barrier")
