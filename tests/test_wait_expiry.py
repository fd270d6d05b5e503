"""Failure detection in the expert kernels' own pipeline waits (needs a GPU).

With moe_test_expert_wait_limit set to 200 ns, the BF16 single-CTA expert kernels give up their waits
for tiles and accumulators long before the data can land: the call returns, the workspace status word
holds a wait timeout (1 or 2; never 3, because the drains of issued copies and MMAs keep the full limit),
and after the workspace is zeroed a normal call on the same GPU matches the oracle with status 0.
The grid-barrier form of the same check is in test_decode_step.py.
"""
import numpy as np
import pytest
import torch

import oracle
import routed_expert_ffn_softmax_gb300 as moe
from test_gpu_parity import DEV, assert_moe_close, small_case, to_np_f32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from routed_expert_ffn_softmax_gb300 import build
    build.build()
    moe.load()
    yield
    moe.moe_test_expert_wait_limit(0)
    moe.moe_set_decode_step_policy(0)


@pytest.mark.parametrize("T,H,I,E,k,skew", [(16, 512, 1024, 8, 2, ()), (40, 256, 512, 4, 2, (0,))])
def test_expert_pipeline_waits_expire_and_the_gpu_recovers(T, H, I, E, k, skew):
    cfg, L, x, lg = small_case(T, H, I, E, k, "bf16", seed=17 + T, skew=skew)
    dev = {n: (v.to(DEV) if v is not None else None) for n, v in L.items()}
    xd, lgd = x.to(DEV), lg.to(DEV)
    ws = moe.alloc_workspace(T, H, I, E, k, moe.MOE_W_BF16, DEV)
    out = torch.empty(T, H, dtype=torch.bfloat16, device=DEV)
    moe.moe_set_decode_step_policy(1)  # the separate launches: the expert kernels run on single CTAs
    try:
        moe.moe_test_expert_wait_limit(200)
        moe.moe_ffn_forward(xd, lgd, dev["W_gate"], dev["W_up"], dev["W_down"], None, None, None, k, out, ws)
        torch.cuda.synchronize()
    finally:
        moe.moe_test_expert_wait_limit(0)
    status = moe.workspace_status(ws)
    assert status in (1, 2), f"expected a wait timeout (1 or 2), got {status}"
    ws.zero_()
    good = torch.full((T, H), float("nan"), dtype=torch.bfloat16, device=DEV)
    moe.moe_ffn_forward(xd, lgd, dev["W_gate"], dev["W_up"], dev["W_down"], None, None, None, k, good, ws)
    torch.cuda.synchronize()
    moe.moe_set_decode_step_policy(0)
    assert moe.workspace_status(ws) == 0
    ref = oracle.forward(x, lg, L["W_gate"], L["W_up"], L["W_down"], top_k=k)
    assert_moe_close(to_np_f32(good), oracle.bf16_bits_to_f32(ref["out"]), "bf16", "after the expired waits")
