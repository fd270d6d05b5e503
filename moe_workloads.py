"""Seeded synthetic workloads for the routed-expert FFN and for decode-phase GQA
attention.

This module is shared by the CUDA path's tests/bench and by the CPU oracle's
tests. It holds only input generation: the expert and attention shapes, the
seeded draws and the offline INT8 weight quantiser that prepares the weights
both sides consume. It holds none of the arithmetic of either operator
(routing, gather, FFN, combine; scores, softmax, weighted sum of values).

Expert shapes and routing top-k come from HiNa-MoE (arXiv 2610.05123),
§8.1 Table 3 ("Expert weight matrix dimensions and routing strategies"):
    Mixtral-8x7B   Gate/Up 4096x14336, Down 14336x4096, Top-2
    Mixtral-8x22B  Gate/Up 6144x16384, Down 16384x6144, Top-2
    DeepSeek-V3    Gate/Up 7168x2048,  Down 2048x7168,  Top-8
    Qwen3-235B     Gate/Up 4096x1536,  Down 1536x4096,  Top-8
Table 3 prints Gate/Up as (hidden x intermediate) in math order; the weights
here are stored the way §2.2 (Figure 3, "general layout") and Algorithm 1's
W(n:n+32, k:k+32) index them: one output row per line, reduction contiguous,
i.e. W_gate/W_up[E, I, H] and W_down[E, H, I].

Expert counts: Mixtral 8, DeepSeek-V3 256, Qwen3-235B 128 (RapidMoE,
arXiv 2610.01265, "Models"). The per-expert token range 1-16 follows HiNa-MoE
§7.3 / Figure 10.

Draws: x ~ N(0,1) -> bf16, router logits ~ N(0,1) f32, weights ~ N(0, 0.02)
-> bf16 (round to nearest even). The INT8 variant quantises those bf16 draws
symmetrically per group of 128 along the reduction dimension (HiNa-MoE §8.1,
"same symmetric group-wise quantization scheme"; group size, scale dtype and
rounding are not printed there, so: scale = max|w|/127 in fp32, q =
clamp(round_half_even(w/scale), -127, 127), and an all-zero group gets scale 1).

Every weight tensor is drawn expert by expert from its own generator, seeded
from (seed, tensor, expert), so one expert's weights never depend on how many
other experts exist or on the device chunking. Draws on CPU and on CUDA use
different torch generators and are not equal to each other: a test draws once
and hands the same tensors to both sides.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, Optional, Sequence, Tuple

import torch

GROUP = 128  # INT8 quantisation group along the reduction dimension


@dataclasses.dataclass(frozen=True)
class MoEConfig:
    name: str
    H: int            # hidden size (gate/up reduction, down output rows)
    I: int            # intermediate size (gate/up output rows, down reduction)
    E: int            # routed experts
    top_k: int
    wtype: str        # "bf16", "int8" or "int8_residual" (gate/up as W^Q + W^R, both INT8)
    T: Tuple[int, ...]  # token counts the workload is run at
    skew_experts: Tuple[int, ...] = ()
    skew: float = 0.0
    seed: int = 0

    @property
    def weight_bytes_per_expert(self) -> int:
        """Algorithmic weight-stream bytes of one expert (3 matrices + scales; the residual split
        streams gate and up twice: W^Q and W^R)."""
        if self.wtype == "bf16":
            return 3 * self.H * self.I * 2
        gu = 2 if self.wtype == "int8_residual" else 1  # streams of gate and of up
        return (2 * gu + 1) * self.H * self.I + 4 * (2 * gu * self.I * (self.H // GROUP) + self.H * (self.I // GROUP))


CONFIGS: Dict[str, MoEConfig] = {
    c.name: c
    for c in (
        MoEConfig("tiny", 256, 512, 8, 2, "bf16", (8,)),
        MoEConfig("mixtral8x7b", 4096, 14336, 8, 2, "bf16", (1, 2, 4, 8, 16, 32, 64)),
        MoEConfig("mixtral8x22b", 6144, 16384, 8, 2, "bf16", (1, 4, 16, 64)),
        # "a skewed variant adding +2.0 to two fixed experts' logits": the two
        # experts are not named; this build takes experts 0 and 1.
        MoEConfig("mixtral8x22b_skew", 6144, 16384, 8, 2, "bf16", (1, 4, 16, 64),
                  skew_experts=(0, 1), skew=2.0),
        MoEConfig("dsv3", 7168, 2048, 256, 8, "bf16", (1, 16, 128, 512)),
        # Prefill-sized batches of the Mixtral-8x7B expert shape (the pages run prefill at 2K-32K
        # tokens, HiNa-MoE §8.2 "Prefill Phase", Table 4): 64 to 1024 tokens per expert, where the
        # expert FFN is a real contraction and is timed in TFLOP/s.
        MoEConfig("mixtral8x7b_prefill", 4096, 14336, 8, 2, "bf16", (256, 1024, 2048, 4096)),
        # The DeepSeek-V3 expert shape at prefill sizes: 128 and 256 tokens per expert over 256 experts.
        MoEConfig("dsv3_prefill", 7168, 2048, 256, 8, "bf16", (4096, 8192)),
        MoEConfig("qwen3_int8", 4096, 1536, 128, 8, "int8", (1, 8, 64, 256)),
        MoEConfig("qwen3_int8_residual", 4096, 1536, 128, 8, "int8_residual", (1, 8, 64, 256)),
    )
}

# tensor ids for generator seeding
_X, _LOGITS, _WG, _WU, _WD = 0, 1, 2, 3, 4


def _gen(device, seed: int, tensor: int, expert: int = 0) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed((seed * 1_000_003 + tensor * 65_537 + expert * 7919 + 12345) % (2**63 - 1))
    return g


def draw_x(T: int, H: int, seed: int = 0, device="cpu") -> torch.Tensor:
    g = _gen(device, seed, _X)
    return torch.randn(T, H, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)


def draw_logits(T: int, E: int, seed: int = 0, device="cpu",
                skew_experts: Sequence[int] = (), skew: float = 0.0) -> torch.Tensor:
    g = _gen(device, seed, _LOGITS)
    lg = torch.randn(T, E, generator=g, device=device, dtype=torch.float32)
    for e in skew_experts:
        lg[:, e] += skew
    return lg


def draw_expert_weight(rows: int, K: int, seed: int, tensor: int, expert: int,
                       device="cpu", std: float = 0.02) -> torch.Tensor:
    g = _gen(device, seed, tensor, expert)
    w = torch.randn(rows, K, generator=g, device=device, dtype=torch.float32)
    return (w * std).to(torch.bfloat16)


def draw_weights(E: int, rows: int, K: int, seed: int, tensor: int, device="cpu",
                 experts: Optional[Sequence[int]] = None) -> torch.Tensor:
    """[len(experts) or E, rows, K] bf16, drawn expert by expert."""
    ids = range(E) if experts is None else experts
    out = torch.empty(len(ids), rows, K, device=device, dtype=torch.bfloat16)
    for n, e in enumerate(ids):
        out[n] = draw_expert_weight(rows, K, seed, tensor, e, device)
    return out


def quantize_int8_groupwise(w: torch.Tensor) -> Tuple[torch.Tensor, torch.Tensor]:
    """Offline weight preparation: bf16 [..., rows, K] -> (int8 q, fp32 scale[..., rows, K/128]).

    Symmetric per-group quantisation along the last (reduction) axis.
    """
    K = w.shape[-1]
    if K % GROUP:
        raise ValueError(f"reduction length {K} is not a multiple of {GROUP}")
    wf = w.float().reshape(*w.shape[:-1], K // GROUP, GROUP)
    s = wf.abs().amax(dim=-1) / 127.0
    zero = s == 0
    s = torch.where(zero, torch.ones_like(s), s)
    q = torch.round(wf / s.unsqueeze(-1)).clamp_(-127, 127)
    q = torch.where(zero.unsqueeze(-1), torch.zeros_like(q), q)
    return q.to(torch.int8).reshape(w.shape), s.contiguous()


def quantize_int8_residual(w: torch.Tensor):
    """Residual-split preparation (RapidMoE, arXiv 2610.01265, "Residual-Split Representation"):
    W^Q = the group-128 INT8 quantisation of w, W^R = the group-128 INT8 quantisation of the fp32
    residual w - W^Q (the pages give no bit width; both parts are INT8 here).
    Returns (qQ int8, sQ fp32, qR int8, sR fp32), scales [..., rows, K/128]."""
    qQ, sQ = quantize_int8_groupwise(w)
    K = w.shape[-1]
    deq = (qQ.float().reshape(*w.shape[:-1], K // GROUP, GROUP) * sQ.unsqueeze(-1)).reshape(w.shape)
    qR, sR = quantize_int8_groupwise(w.float() - deq)
    return qQ, sQ, qR, sR


def make_layer(cfg: MoEConfig, seed: Optional[int] = None, device="cpu",
               experts: Optional[Sequence[int]] = None) -> Dict[str, torch.Tensor]:
    """Expert weights of one MoE layer: W_gate/W_up [E,I,H], W_down [E,H,I] (+ INT8 scales).

    For INT8 the returned W_* are int8 and s_* hold the fp32 group scales
    (s_gate/s_up [E,I,H/128], s_down [E,H,I/128]); for BF16 s_* are None. The residual split
    adds Wr_gate/Wr_up (int8 residual parts) and sr_gate/sr_up (their scales).
    """
    seed = cfg.seed if seed is None else seed
    wg = draw_weights(cfg.E, cfg.I, cfg.H, seed, _WG, device, experts)
    wu = draw_weights(cfg.E, cfg.I, cfg.H, seed, _WU, device, experts)
    wd = draw_weights(cfg.E, cfg.H, cfg.I, seed, _WD, device, experts)
    if cfg.wtype == "bf16":
        return dict(W_gate=wg, W_up=wu, W_down=wd, s_gate=None, s_up=None, s_down=None)
    if cfg.wtype == "int8_residual":
        qg, sg, rg, srg = quantize_int8_residual(wg)
        del wg
        qu, su, ru, sru = quantize_int8_residual(wu)
        del wu
        qd, sd = quantize_int8_groupwise(wd)
        del wd
        return dict(W_gate=qg, W_up=qu, W_down=qd, s_gate=sg, s_up=su, s_down=sd,
                    Wr_gate=rg, Wr_up=ru, sr_gate=srg, sr_up=sru)
    qg, sg = quantize_int8_groupwise(wg)
    del wg
    qu, su = quantize_int8_groupwise(wu)
    del wu
    qd, sd = quantize_int8_groupwise(wd)
    del wd
    return dict(W_gate=qg, W_up=qu, W_down=qd, s_gate=sg, s_up=su, s_down=sd)


def make_tokens(cfg: MoEConfig, T: int, seed: Optional[int] = None, device="cpu"):
    """(x [T,H] bf16, router logits [T,E] f32) for one decode step."""
    seed = cfg.seed if seed is None else seed
    x = draw_x(T, cfg.H, seed, device)
    lg = draw_logits(T, cfg.E, seed, device, cfg.skew_experts, cfg.skew)
    return x, lg


# ----------------------------------------------------------------------------
# Decode-phase GQA attention inputs (HiNa-MoE §6.1, Figure 9).
#
# Head counts and head dim are those of the GQA models the pages name: Qwen3-30B-A3B
# (32 query heads, 4 key/value heads: the group of 8 the pages quote), Mixtral-8x7B
# (32 / 8) and Qwen3-235B-A22B (64 / 4); all use d = 128. Sequence lengths: the pages
# run decode after 512-token prompts (RapidMoE, "Datasets and Workloads") and prefill
# at 2K-32K tokens (HiNa-MoE Table 4); a decode batch here mixes lengths drawn
# uniformly from [len_lo, len_hi]. Draws: q, K, V ~ N(0,1) -> bf16; cache rows past a
# sequence's length are filled with NaN, which the attention must never read.

@dataclasses.dataclass(frozen=True)
class AttnConfig:
    name: str
    h_q: int
    h_kv: int
    d: int
    B: int            # sequences in the decode batch (one new token each)
    len_lo: int
    len_hi: int       # also the cache capacity L_cap
    seed: int = 0

    @property
    def group(self) -> int:
        return self.h_q // self.h_kv

    @property
    def scale(self) -> float:
        return 1.0 / float(self.d) ** 0.5


ATTN_CONFIGS: Dict[str, AttnConfig] = {
    c.name: c
    for c in (
        AttnConfig("attn_tiny", 16, 2, 128, 5, 1, 700),
        AttnConfig("qwen3_30b_attn", 32, 4, 128, 64, 512, 8192),
        AttnConfig("mixtral8x7b_attn", 32, 8, 128, 16, 2048, 32768),
        AttnConfig("qwen3_235b_attn", 64, 4, 128, 64, 512, 8192),
    )
}

_AQ, _AK, _AV, _ALEN = 10, 11, 12, 13


def draw_seq_lens(B: int, lo: int, hi: int, seed: int = 0) -> torch.Tensor:
    """[B] int32 sequence lengths, uniform in [lo, hi] (drawn on the CPU)."""
    g = _gen("cpu", seed, _ALEN)
    return torch.randint(lo, hi + 1, (B,), generator=g, dtype=torch.int64).to(torch.int32)


def make_attention(cfg: AttnConfig, seed: Optional[int] = None, device="cpu",
                   seq_lens: Optional[torch.Tensor] = None, L_cap: Optional[int] = None):
    """(q [B,h_q,d], K [B,h_kv,L_cap,d], V [B,h_kv,L_cap,d] bf16, seq_lens [B] int32).

    Rows at or past seq_lens[b] hold NaN."""
    seed = cfg.seed if seed is None else seed
    L_cap = cfg.len_hi if L_cap is None else L_cap
    if seq_lens is None:
        seq_lens = draw_seq_lens(cfg.B, cfg.len_lo, cfg.len_hi, seed)
    B = seq_lens.shape[0]
    q = torch.randn(B, cfg.h_q, cfg.d, generator=_gen(device, seed, _AQ), device=device).to(torch.bfloat16)
    kv = []
    for t in (_AK, _AV):
        m = torch.randn(B, cfg.h_kv, L_cap, cfg.d, generator=_gen(device, seed, t), device=device)
        m = m.to(torch.bfloat16)
        past = torch.arange(L_cap, device=device)[None, :] >= seq_lens.to(device)[:, None].long()
        m.masked_fill_(past[:, None, :, None], float("nan"))
        kv.append(m)
    return q, kv[0], kv[1], seq_lens.to(torch.int32)


def attention_kv_bytes(seq_lens: torch.Tensor, h_kv: int, d: int) -> int:
    """Algorithmic bytes of the key/value rows one decode call must read (bf16)."""
    return int(seq_lens.long().sum()) * h_kv * d * 2 * 2


def expected_active(cfg: MoEConfig, T: int) -> float:
    """E[A] under uniform routing: E * (1 - (1 - k/E)^T)."""
    return cfg.E * (1.0 - (1.0 - cfg.top_k / cfg.E) ** T)
