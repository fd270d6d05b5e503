"""Expert weights resident in host memory (pinned; Grace LPDDR5X on a GB300 node), read by the
same kernels over NVLink-C2C through their device-visible addresses: HiNa-MoE §1 keeps routed
experts in CPU memory when they do not fit the GPU, and §3.1 keeps one general layout that CPU
and GPU both use. The C ABI takes such pointers unchanged; the results must equal the oracle
and be bit-identical to the run with the same weights in HBM (needs a GPU)."""
import numpy as np
import pytest
import torch

import moe_workloads as mw
import oracle
import routed_expert_ffn_softmax_gb300 as moe
from test_gpu_parity import (DEV, assert_moe_close, check_route, gpu_route, oracle_rows, run_forward_ws, small_case,
                             to_np_f32)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from routed_expert_ffn_softmax_gb300 import build
    build.build()
    moe.load()
    yield


def pinned(L):
    return {n: (torch.empty(v.shape, dtype=v.dtype, pin_memory=True).copy_(v) if v is not None else None)
            for n, v in L.items()}


def forward(W, x, lg, k, cfg):
    wt = moe.MOE_W_INT8_G128 if cfg.wtype == "int8" else moe.MOE_W_BF16
    T = x.shape[0]
    ws = moe.alloc_workspace(T, cfg.H, cfg.I, cfg.E, k, wt, DEV)
    out = torch.full((T, cfg.H), float("nan"), dtype=torch.bfloat16, device=DEV)
    moe.moe_ffn_forward(x.to(DEV), lg.to(DEV), W["W_gate"], W["W_up"], W["W_down"], W["s_gate"], W["s_up"],
                        W["s_down"], k, out, ws)
    torch.cuda.synchronize()
    assert moe.workspace_status(ws) == 0
    return out


@pytest.mark.parametrize("T,H,I,E,k,wtype,skew", [
    (8, 256, 512, 8, 2, "bf16", ()),
    (150, 64, 256, 4, 2, "bf16", (0, 1)),   # several passes per expert
    (70, 384, 256, 8, 4, "int8", (2,)),     # CTA-pair kernels, half-empty last row block
    (2, 256, 512, 8, 2, "bf16", ()),        # about one token per expert
    (4, 256, 384, 16, 4, "int8", ()),
])
def test_host_weights_match_oracle_and_device_run(T, H, I, E, k, wtype, skew):
    cfg, L, x, lg = small_case(T, H, I, E, k, wtype, seed=5 * T + H, skew=skew)
    out_host = forward(pinned(L), x, lg, k, cfg)
    out_dev, _ = run_forward_ws(L, x, lg, k)
    assert torch.equal(out_host, out_dev)
    ref = oracle.forward(x, lg, L["W_gate"], L["W_up"], L["W_down"], L["s_gate"], L["s_up"], L["s_down"],
                         wtype=wtype, top_k=k)
    assert_moe_close(to_np_f32(out_host), oracle.bf16_bits_to_f32(ref["out"]), wtype, f"host weights T={T}")


@pytest.mark.parametrize("name,T", [("mixtral8x7b", 16), ("qwen3_int8", 8)])
def test_host_weights_full_size_every_token(name, T):
    cfg = mw.CONFIGS[name]
    Lg = mw.make_layer(cfg, device=DEV)
    Lh = pinned(Lg)
    x, lg = mw.make_tokens(cfg, T, device=DEV)
    got = to_np_f32(forward(Lh, x, lg, cfg.top_k, cfg))
    assert np.all(np.isfinite(got))
    ro, rows = oracle_rows(cfg, Lh, x.cpu(), lg.cpu())  # the pinned copy is the oracle's CPU layer
    for t in range(T):
        assert_moe_close(got[t], rows[t], cfg.wtype, f"{name} T={T} token {t} (host weights)")
    check_route(gpu_route(lg, cfg.top_k), ro)
    del Lg, Lh
    torch.cuda.empty_cache()
