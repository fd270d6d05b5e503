"""Pins of the decode GQA attention oracle to things other than itself (no GPU).

HiNa-MoE (arXiv 2610.05123) §6.1 / Figure 9 defines the operator: per key/value head, a
small block of G = h_q / h_kv query heads times the l_seq x d key head, then the
probabilities times the value head. Each test checks the oracle against a fact fixed
outside it: hand-worked fixtures, torch's own scaled_dot_product_attention (a library
routine, float64 on the CPU), closed forms (one key, equal keys, zero query, one dominating
key, an empty sequence) and invariants (key permutation, cache contents past the length,
which key/value head a query head reads).
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


def as_bf16(a) -> torch.Tensor:
    return torch.tensor(np.asarray(a, dtype=np.float64), dtype=torch.float32).to(torch.bfloat16)


def run(q, k, v, lens, scale):
    return oracle.gqa_decode(q, k, v, torch.as_tensor(lens, dtype=torch.int32), scale)


def case(cfg_name="attn_tiny", seed=0, lens=None, L_cap=None, **kw):
    cfg = mw.ATTN_CONFIGS[cfg_name]
    if kw:
        import dataclasses
        cfg = dataclasses.replace(cfg, **kw)
    lt = None if lens is None else torch.tensor(lens, dtype=torch.int32)
    return cfg, mw.make_attention(cfg, seed=seed, seq_lens=lt, L_cap=L_cap)


# ----------------------------------------------------------------------------
def test_golden_worked_examples():
    with open(os.path.join(GOLDEN, "gqa_worked.json")) as f:
        fx = json.load(f)
    assert "§6.1" in fx["citation"]
    for c in fx["cases"]:
        conv = lambda a: np.vectorize(lambda x: np.nan if x == "nan" else float(x), otypes=[np.float64])(
            np.array(a, dtype=object))
        q, k, v = as_bf16(conv(c["q"])), as_bf16(conv(c["K"])), as_bf16(conv(c["V"]))
        assert q.shape[1] == c["h_q"] and k.shape[1] == c["h_kv"] and k.shape[2] == c["L_cap"]
        r = run(q, k, v, c["seq_lens"], c["scale_f32"])
        want = np.array(c["out"], dtype=np.float64)
        np.testing.assert_allclose(r["out_f64"], want, rtol=0, atol=1e-6, err_msg=c["name"])
        assert np.array_equal(r["out"], bits(as_bf16(want))), c["name"]


def sdpa_reference(q, k, v, lens, scale):
    """torch.nn.functional.scaled_dot_product_attention in float64, one sequence at a time,
    key/value heads repeated G times along the head axis (consecutive query heads share)."""
    B, h_q, d = q.shape
    h_kv = k.shape[1]
    G = h_q // h_kv
    out = np.zeros((B, h_q, d), np.float64)
    for b in range(B):
        n = int(lens[b])
        if n == 0:
            continue
        kb = k[b, :, :n].double().repeat_interleave(G, dim=0)[None]
        vb = v[b, :, :n].double().repeat_interleave(G, dim=0)[None]
        qb = q[b].double()[None, :, None, :]
        out[b] = torch.nn.functional.scaled_dot_product_attention(qb, kb, vb, scale=scale)[0, :, 0].numpy()
    return out


@pytest.mark.parametrize("h_q,h_kv,d,lens", [
    (16, 2, 128, (510, 1, 129, 128, 700)),
    (8, 8, 64, (3, 40)),      # G = 1 (multi-head)
    (12, 3, 32, (17, 0, 5)),  # G = 4, an empty sequence
    (16, 1, 16, (300,)),      # one key/value head for all query heads
])
def test_matches_library_sdpa(h_q, h_kv, d, lens):
    cfg, (q, k, v, ln) = case(lens=lens, L_cap=max(lens) + 3, h_q=h_q, h_kv=h_kv, d=d, seed=len(lens))
    r = run(q, k, v, ln, cfg.scale)
    ref = sdpa_reference(q, k, v, ln, float(np.float32(cfg.scale)))  # the ABI takes the scale as float32
    np.testing.assert_allclose(r["out_f64"], ref, rtol=1e-10, atol=1e-12)
    assert np.array_equal(r["out"], oracle.f64_to_bf16_bits(ref))


def test_one_key_returns_that_value_row():
    cfg, (q, k, v, ln) = case(lens=(1, 1, 1), L_cap=4)
    r = run(q, k, v, ln, cfg.scale)
    G = cfg.group
    for b in range(3):
        for h in range(cfg.h_q):
            assert np.array_equal(r["out"][b, h], bits(v[b, h // G, 0]))


def test_equal_keys_and_zero_query_average_the_values():
    cfg, (q, k, v, ln) = case(lens=(37, 250), L_cap=256)
    k_eq = k.clone()
    k_eq[:, :, :] = k[:, :, :1]                          # every key row equal
    q0 = torch.zeros_like(q)
    G = cfg.group
    for qq, kk in ((q, k_eq), (q0, k)):
        r = run(qq, kk, v, ln, cfg.scale)
        for b, n in enumerate(ln.tolist()):
            mean = v[b, :, :n].double().mean(dim=1).numpy()          # [h_kv, d]
            np.testing.assert_allclose(r["out_f64"][b], np.repeat(mean, G, axis=0), rtol=1e-12, atol=1e-14)


def test_dominating_key_selects_its_value():
    cfg, (q, k, v, ln) = case(lens=(90,), L_cap=96, h_q=2, h_kv=1)
    k = k.clone()
    q = torch.zeros_like(q)
    q[0, :, 0] = 1.0
    k[0, 0, :90, :] = 0.0
    k[0, 0, 41, 0] = 8192.0                               # score 8192 * scale = 724 above all others
    r = run(q, k, v, ln, cfg.scale)
    for h in range(2):
        assert np.array_equal(r["out"][0, h], bits(v[0, 0, 41]))


def test_key_permutation_invariance():
    cfg, (q, k, v, ln) = case(lens=(300, 77), L_cap=320)
    r0 = run(q, k, v, ln, cfg.scale)
    k2, v2 = k.clone(), v.clone()
    g = torch.Generator().manual_seed(3)
    for b, n in enumerate(ln.tolist()):
        perm = torch.randperm(n, generator=g)
        k2[b, :, :n] = k[b, :, perm]
        v2[b, :, :n] = v[b, :, perm]
    r1 = run(q, k2, v2, ln, cfg.scale)
    np.testing.assert_allclose(r1["out_f64"], r0["out_f64"], rtol=1e-12, atol=1e-14)


def test_cache_past_length_is_never_read():
    cfg, (q, k, v, ln) = case(lens=(5, 64, 129), L_cap=200)
    r0 = run(q, k, v, ln, cfg.scale)
    k2, v2 = k.clone(), v.clone()
    for b, n in enumerate(ln.tolist()):
        k2[b, :, n:] = 1e30
        v2[b, :, n:] = -3.0
    r1 = run(q, k2, v2, ln, cfg.scale)
    assert np.array_equal(r1["out"], r0["out"]) and np.array_equal(r1["out_f64"], r0["out_f64"])
    assert np.all(np.isfinite(r0["out_f64"]))


def test_query_head_reads_key_value_head_of_its_group():
    """Query head hq reads key/value head hq // G: changing key/value head j changes exactly
    the query heads j*G .. j*G+G-1."""
    cfg, (q, k, v, ln) = case(lens=(60, 61), L_cap=64, h_q=12, h_kv=3)
    G = cfg.group
    r0 = run(q, k, v, ln, cfg.scale)
    for j in range(3):
        v2 = v.clone()
        v2[:, j] = v2[:, j] * 2.0                        # exact in bf16
        r1 = run(q, k, v2, ln, cfg.scale)
        changed = np.any(r1["out_f64"] != r0["out_f64"], axis=(0, 2))
        assert changed.tolist() == [hq // G == j for hq in range(12)]
        np.testing.assert_allclose(r1["out_f64"][:, j * G:(j + 1) * G], 2 * r0["out_f64"][:, j * G:(j + 1) * G],
                                   rtol=1e-12, atol=1e-14)


def test_empty_sequence_gives_zero_and_bad_lengths_are_rejected():
    cfg, (q, k, v, ln) = case(lens=(0, 3), L_cap=8)
    r = run(q, k, v, ln, cfg.scale)
    assert not r["out"][0].any() and not r["out_f64"][0].any()
    with pytest.raises(ValueError):
        run(q, k, v, (9, 3), cfg.scale)
    with pytest.raises(ValueError):
        run(q, k, v, (-1, 3), cfg.scale)


def test_double_to_bf16_rounding():
    """The oracle rounds float64 to bf16 once (ties to even), not through float32."""
    one_ulp = 2.0 ** -7
    vals = np.array([1.0 + one_ulp / 2,                   # tie -> even (1.0)
                     1.0 + 3 * one_ulp / 2,               # tie -> even (1 + 2 ulp)
                     1.0 + one_ulp / 2 + 2.0 ** -40,      # just above the tie: float32 would round to the tie
                     -2.5, 0.0, 3.3895313892515355e38, 3.5e38, 2.0 ** -133, 2.0 ** -135])
    got = oracle.f64_to_bf16_bits(vals)
    want = [0x3F80, 0x3F82, 0x3F81, 0xC020, 0x0000, 0x7F7F, 0x7F80, 0x0001, 0x0000]
    assert got.tolist() == want
    # the same values through numpy's float32 then bf16 (double rounding) differ at the 3rd entry
    assert bits(torch.tensor(vals[2:3], dtype=torch.float64).to(torch.float32).to(torch.bfloat16))[0] == 0x3F80
