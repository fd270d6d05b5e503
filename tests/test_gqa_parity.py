"""Decode GQA attention on the GPU (moe_gqa_decode, through the C ABI) against the CPU oracle
(needs a GPU).

HiNa-MoE (arXiv 2610.05123) §6.1, Figure 9. Tolerance, from the kernel's arithmetic: the
probabilities enter the probability x value product rounded to bf16 (relative error <= 2^-8
each) and the output is rounded to bf16 once (<= 2^-8 |o|). Per output element,
    |gpu - o| <= 2^-8 * sum_i p_i |v_i| + 2^-8 * |o| + slack,
where sum_i p_i |v_i| is the oracle's attention over |V| (computed exactly, float64), and the
slack 2^-12 * sum_i p_i |v_i| + 1e-6 covers the fp32 scores (bf16 products, fp32 sums of 128),
the approximate 2^x (relative error about 2^-22) and the fp32 accumulation over tiles and pieces. A wrong key/value head, a transposed
operand or a lost tile changes outputs by about |o| itself, far above this bound for the
random inputs here.
"""
import dataclasses

import numpy as np
import pytest
import torch

import moe_workloads as mw
import oracle
import routed_expert_ffn_softmax_gb300 as moe

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _built():
    from routed_expert_ffn_softmax_gb300 import build
    build.build()
    moe.load()
    yield


def gpu_decode(q, k, v, lens, scale, ws=None):
    B, h_q, d = q.shape
    h_kv, L_cap = k.shape[1], k.shape[2]
    if ws is None:
        ws = moe.alloc_gqa_workspace(B, h_q, h_kv, d, L_cap, DEV)
    out = torch.full((B, h_q, d), float("nan"), dtype=torch.bfloat16, device=DEV)
    moe.moe_gqa_decode(q.to(DEV), k.to(DEV), v.to(DEV), lens.to(DEV), scale, out, ws)
    torch.cuda.synchronize()
    return out, moe.workspace_status(ws)


def bound_check(got, q, k, v, lens, scale, what):
    """got: GPU output [B,h_q,d] (any device); inputs on the CPU."""
    ref = oracle.gqa_decode(q, k, v, lens, scale)["out_f64"]
    v_abs = v.abs()
    v_abs = torch.where(torch.isnan(v_abs), torch.zeros_like(v_abs), v_abs)  # rows past the lengths
    ref_abs = oracle.gqa_decode(q, k, v_abs, lens, scale)["out_f64"]
    g = got.float().cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(g)), f"{what}: non-finite output"
    tol = (2.0 ** -8 + 2.0 ** -12) * ref_abs + 2.0 ** -8 * np.abs(ref) + 1e-6
    err = np.abs(g - ref)
    bad = err > tol
    assert not bad.any(), (f"{what}: {bad.sum()} elements out of bound; worst at "
                           f"{np.unravel_index(np.argmax(err - tol), err.shape)}: err {err.max():.3g}")
    return err, ref


def attn_case(h_q, h_kv, lens, L_cap, seed=0):
    cfg = dataclasses.replace(mw.ATTN_CONFIGS["attn_tiny"], h_q=h_q, h_kv=h_kv)
    q, k, v, ln = mw.make_attention(cfg, seed=seed, seq_lens=torch.tensor(lens, dtype=torch.int32), L_cap=L_cap)
    return cfg, q, k, v, ln


@pytest.mark.parametrize("h_q,h_kv,lens,L_cap", [
    (16, 2, (510, 586, 566, 47, 615), 700),          # the tiny workload: G = 8
    (32, 4, (1, 127, 128, 129, 255, 256, 257), 300),  # tile edges, G = 8
    (32, 8, (1000, 3, 64), 1000),                    # G = 4 (Mixtral), L_cap not a multiple of 128
    (64, 4, (333, 900), 1024),                       # G = 16 (Qwen3-235B)
    (8, 8, (200, 1), 256),                           # G = 1
    (4, 2, (77,), 77),                               # G = 2, L_cap = length
    (12, 4, (150, 260), 300),                        # G = 3: padded to 4
    (24, 2, (400,), 512),                            # G = 12: padded to 16
])
def test_matches_oracle(h_q, h_kv, lens, L_cap):
    cfg, q, k, v, ln = attn_case(h_q, h_kv, lens, L_cap, seed=h_q + len(lens))
    out, st = gpu_decode(q, k, v, ln, cfg.scale)
    assert st == 0
    bound_check(out, q, k, v, ln, cfg.scale, f"h_q={h_q} h_kv={h_kv} lens={lens}")


def test_segments_split_across_many_ctas():
    """One long sequence with one key/value head: its ~160 tiles are spread over every CTA, so
    the output is merged from one piece per CTA; plus short sequences around it."""
    cfg, q, k, v, ln = attn_case(8, 1, (5, 20000, 130, 1), 20096, seed=7)
    out, st = gpu_decode(q, k, v, ln, cfg.scale)
    assert st == 0
    bound_check(out, q, k, v, ln, cfg.scale, "long sequence split")


def test_many_short_sequences():
    lens = tuple(int(x) for x in torch.randint(1, 300, (300,), generator=torch.Generator().manual_seed(1)))
    cfg, q, k, v, ln = attn_case(32, 4, lens, 300, seed=3)
    out, st = gpu_decode(q, k, v, ln, cfg.scale)
    assert st == 0
    bound_check(out, q, k, v, ln, cfg.scale, "300 short sequences")


def test_empty_and_invalid_lengths():
    cfg, q, k, v, ln = attn_case(32, 4, (0, 200, 0, 129), 256, seed=11)
    out, st = gpu_decode(q, k, v, ln, cfg.scale)
    assert st == 0
    assert torch.count_nonzero(out[0].float()) == 0 and torch.count_nonzero(out[2].float()) == 0
    bound_check(out, q, k, v, ln, cfg.scale, "empty sequences")
    # a length past the cache capacity: reported in the status word, that sequence gets 0
    ws = moe.alloc_gqa_workspace(4, 32, 4, 128, 256, DEV)
    bad = ln.clone()
    bad[1] = 257
    out2, st2 = gpu_decode(q, k, v, bad, cfg.scale, ws)
    assert st2 == 4
    assert torch.count_nonzero(out2[1].float()) == 0
    bound_check(out2[3:4], q[3:4], k[3:4], v[3:4], ln[3:4], cfg.scale, "beside a bad length")
    # the status is sticky; the workspace stays usable, and zeroing the word resets it
    out3, st3 = gpu_decode(q, k, v, ln, cfg.scale, ws)
    assert st3 == 4 and torch.equal(out3, out)
    ws[:4] = 0
    out4, st4 = gpu_decode(q, k, v, ln, cfg.scale, ws)
    assert st4 == 0 and torch.equal(out4, out)


def test_deterministic_and_workspace_reuse():
    cfg, q, k, v, ln = attn_case(32, 4, (3000, 17, 1500), 3072, seed=5)
    ws = moe.alloc_gqa_workspace(3, 32, 4, 128, 3072, DEV)
    a, _ = gpu_decode(q, k, v, ln, cfg.scale, ws)
    b, _ = gpu_decode(q, k, v, ln, cfg.scale, ws)
    assert torch.equal(a, b)


def test_softmax_scale_and_dominating_key():
    """A key whose score dwarfs the rest gets all the weight: output = its value row (bf16-exact)."""
    cfg, q, k, v, ln = attn_case(16, 2, (700, 300), 704, seed=2)
    k = k.clone()
    q = q.clone()
    q[:, :, :] = 0.0
    q[:, :, 5] = 1.0
    k[:, :, :, 5] = 0.0
    k[0, 1, 433, 5] = 4096.0
    k[1, 0, 0, 5] = 4096.0
    out, st = gpu_decode(q, k, v, ln, 1.0)
    assert st == 0
    for h in range(8, 16):
        assert torch.equal(out[0, h].cpu(), v[0, 1, 433])
    for h in range(8):
        assert torch.equal(out[1, h].cpu(), v[1, 0, 0])


@pytest.mark.parametrize("name", ["qwen3_30b_attn", "mixtral8x7b_attn", "qwen3_235b_attn"])
def test_full_size_sampled(name):
    """The bench's workloads at full size on the GPU; the oracle checks three whole sequences."""
    cfg = mw.ATTN_CONFIGS[name]
    q, k, v, ln = mw.make_attention(cfg, device=DEV)
    out, st = gpu_decode(q, k, v, ln, cfg.scale)
    assert st == 0
    for b in sorted({0, cfg.B // 2, cfg.B - 1}):
        n = int(ln[b])
        qb, kb, vb = q[b:b + 1].cpu(), k[b:b + 1, :, :n].cpu(), v[b:b + 1, :, :n].cpu()
        bound_check(out[b:b + 1], qb, kb, vb, ln[b:b + 1].cpu(), cfg.scale, f"{name} sequence {b} (len {n})")
    del q, k, v
    torch.cuda.empty_cache()
