"""Routed-expert MoE FFN and decode GQA attention for the GB300 (sm_103a): Python binding of
libmoe.so.

Every function here has the name of the C entry point it calls (include/moe.h,
include/moe_gqa.h)
and only marshals arguments: torch tensors in, device pointers and sizes out.
All arithmetic runs in the library's CUDA kernels. There is no fallback: if
libmoe.so is missing or cannot be loaded, importing the binding's functions
raises.

Build the library with ``routed_expert_ffn_softmax_gb300.build.build()``.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

from . import build as _build

__all__ = [
    "MoeError", "MOE_W_BF16", "MOE_W_INT8_G128", "load", "lib_path",
    "moe_status_string", "moe_workspace_size", "moe_route_topk", "moe_gather",
    "moe_expert_ffn", "moe_combine", "moe_ffn_forward", "alloc_workspace", "workspace_status",
    "moe_expert_ffn_noalloc", "moe_expert_ffn_noalloc_status", "moe_gqa_workspace_size", "moe_gqa_decode", "alloc_gqa_workspace",
    "moe_expert_ffn_residual", "moe_ffn_forward_residual", "moe_set_decode_step_policy", "moe_ffn_forward_launches",
    "moe_test_expire_grid_barrier", "moe_set_expert_pass_tokens", "moe_test_expert_wait_limit",
]

MOE_W_BF16 = 0
MOE_W_INT8_G128 = 1

_STATUS = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED", 3: "MOE_ERR_WORKSPACE",
           4: "MOE_ERR_CUDA"}

_lock = threading.Lock()
_lib: Optional[ctypes.CDLL] = None


class MoeError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} returned {_STATUS.get(status, status)}")


def lib_path() -> str:
    return _build.LIB


def load() -> ctypes.CDLL:
    """Load libmoe.so; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_build.LIB):
            raise ImportError(f"{_build.LIB} not found: build it with routed_expert_ffn_softmax_gb300.build.build()")
        lib = ctypes.CDLL(_build.LIB)
        P, i, z = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
        lib.moe_status_string.argtypes = [i]
        lib.moe_status_string.restype = ctypes.c_char_p
        lib.moe_workspace_size.argtypes = [i, i, i, i, i, i]
        lib.moe_workspace_size.restype = z
        lib.moe_route_topk.argtypes = [P, i, i, i, P, P, P, P, P, P, P, P, P]
        lib.moe_gather.argtypes = [P, i, i, i, P, P, P]
        lib.moe_expert_ffn.argtypes = [P, P, P, P, P, P, P, P, P, P, i, i, i, i, i, P, P, z, P]
        lib.moe_combine.argtypes = [P, P, P, i, i, i, P, P]
        lib.moe_ffn_forward.argtypes = [P, P, P, P, P, P, P, P, i, i, i, i, i, i, P, P, z, P]
        lib.moe_expert_ffn_residual.argtypes = [P] * 14 + [i, i, i, i, P, P, z, P]
        lib.moe_ffn_forward_residual.argtypes = [P] * 12 + [i, i, i, i, i, P, P, z, P]
        lib.moe_gqa_workspace_size.argtypes = [i, i, i, i, i]
        lib.moe_gqa_workspace_size.restype = z
        lib.moe_gqa_decode.argtypes = [P, P, P, P, i, i, i, i, i, ctypes.c_float, P, P, z, P]
        lib.moe_set_decode_step_policy.argtypes = [i]
        lib.moe_ffn_forward_launches.argtypes = [i, i, i, i, i, i]
        for f in ("moe_set_decode_step_policy", "moe_ffn_forward_launches"):
            getattr(lib, f).restype = i
        for f in ("moe_route_topk", "moe_gather", "moe_expert_ffn", "moe_combine", "moe_ffn_forward",
                  "moe_gqa_decode", "moe_expert_ffn_residual", "moe_ffn_forward_residual"):
            getattr(lib, f).restype = i
        _lib = lib
        return lib


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensors passed to libmoe must be contiguous")
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _check(fn: str, status: int) -> None:
    if status != 0:
        raise MoeError(fn, status)


def _wtype(W: torch.Tensor) -> int:
    if W.dtype == torch.int8:
        return MOE_W_INT8_G128
    if W.dtype == torch.bfloat16:
        return MOE_W_BF16
    raise TypeError(f"expert weights must be bf16 or int8, got {W.dtype}")


def moe_status_string(status: int) -> str:
    return load().moe_status_string(status).decode()


def moe_workspace_size(T: int, H: int, I: int, E: int, top_k: int, wtype: int = MOE_W_BF16) -> int:
    return int(load().moe_workspace_size(T, H, I, E, top_k, wtype))


def alloc_workspace(T, H, I, E, top_k, wtype=MOE_W_BF16, device="cuda") -> torch.Tensor:
    """A zero-filled workspace (it must start zeroed; calls leave it reusable)."""
    n = moe_workspace_size(T, H, I, E, top_k, wtype)
    if n == 0:
        raise ValueError("invalid sizes for moe_workspace_size")
    return torch.zeros(n, dtype=torch.uint8, device=device)


def workspace_status(workspace: torch.Tensor) -> int:
    """The status word kernels leave in the workspace (0 = no kernel gave up a wait)."""
    return int(workspace[:4].view(torch.int32).item())


def moe_route_topk(logits, top_k, topk_ids, topk_w, expert_counts, expert_offsets, sorted_token, inv_pos,
                   active_experts, num_active, stream=None) -> None:
    T, E = logits.shape
    _check("moe_route_topk", load().moe_route_topk(
        _ptr(logits), T, E, top_k, _ptr(topk_ids), _ptr(topk_w), _ptr(expert_counts), _ptr(expert_offsets),
        _ptr(sorted_token), _ptr(inv_pos), _ptr(active_experts), _ptr(num_active), _stream(stream)))


def moe_gather(x, top_k, sorted_token, xg, stream=None) -> None:
    T, H = x.shape
    _check("moe_gather", load().moe_gather(_ptr(x), T, H, top_k, _ptr(sorted_token), _ptr(xg), _stream(stream)))


def moe_expert_ffn(xg, expert_offsets, active_experts, num_active, W_gate, W_up, W_down, s_gate, s_up, s_down,
                   Y, workspace, stream=None) -> None:
    P, H = xg.shape
    E, I, _ = W_gate.shape
    _check("moe_expert_ffn", load().moe_expert_ffn(
        _ptr(xg), _ptr(expert_offsets), _ptr(active_experts), _ptr(num_active), _ptr(W_gate), _ptr(W_up),
        _ptr(W_down), _ptr(s_gate), _ptr(s_up), _ptr(s_down), _wtype(W_gate), H, I, E, P, _ptr(Y),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)))


def moe_combine(Y, inv_pos, topk_w, top_k, out, stream=None) -> None:
    T, H = out.shape
    _check("moe_combine", load().moe_combine(_ptr(Y), _ptr(inv_pos), _ptr(topk_w), T, top_k, H, _ptr(out),
                                             _stream(stream)))


def moe_ffn_forward(x, logits, W_gate, W_up, W_down, s_gate, s_up, s_down, top_k, out, workspace,
                    stream=None) -> None:
    T, H = x.shape
    E, I, _ = W_gate.shape
    _check("moe_ffn_forward", load().moe_ffn_forward(
        _ptr(x), _ptr(logits), _ptr(W_gate), _ptr(W_up), _ptr(W_down), _ptr(s_gate), _ptr(s_up), _ptr(s_down),
        _wtype(W_gate), T, H, I, E, top_k, _ptr(out), _ptr(workspace), workspace.numel() * workspace.element_size(),
        _stream(stream)))


def moe_set_decode_step_policy(policy: int) -> None:
    """0: by batch shape (default: the one-launch decode step for INT8 with 2 * T * top_k <= E and BF16 with T <= 2); 1: never; 2: whenever
    the sizes allow."""
    _check("moe_set_decode_step_policy", load().moe_set_decode_step_policy(policy))


def moe_set_expert_pass_tokens(gate_up: int = 0, down: int = 0) -> None:
    """Tokens per pass of the BF16 expert kernels (64, 128, 192 or 256; 0 = by batch shape, the default).
    Size workspaces after setting it (see include/moe.h)."""
    f = load().moe_set_expert_pass_tokens
    f.argtypes = [ctypes.c_int, ctypes.c_int]
    f.restype = ctypes.c_int
    _check("moe_set_expert_pass_tokens", f(int(gate_up), int(down)))


def moe_test_expert_wait_limit(wait_ns: int = 0) -> None:
    """Failure-detection test hook: limit of the BF16 single-CTA expert kernels' pipeline waits (ns; 0 =
    the normal 2 s). A short limit makes the waits run out: nonzero workspace status (see include/moe.h)."""
    f = load().moe_test_expert_wait_limit
    f.argtypes = [ctypes.c_uint64]
    f.restype = ctypes.c_int
    _check("moe_test_expert_wait_limit", f(int(wait_ns)))


def moe_test_expire_grid_barrier(enable: bool, wait_ns: int = 2_000_000_000) -> None:
    """Failure-detection test hook: the one-launch decode step's grid barrier never opens while enabled
    and every CTA gives up after wait_ns (status 5 in the workspace; see include/moe.h)."""
    f = load().moe_test_expire_grid_barrier
    f.argtypes = [ctypes.c_int, ctypes.c_uint64]
    f.restype = ctypes.c_int
    _check("moe_test_expire_grid_barrier", f(1 if enable else 0, int(wait_ns)))


def moe_ffn_forward_launches(T, H, I, E, top_k, wtype=MOE_W_BF16) -> int:
    """Kernels one moe_ffn_forward call launches for these sizes under the current policy."""
    return int(load().moe_ffn_forward_launches(T, H, I, E, top_k, wtype))


def moe_expert_ffn_noalloc(xg, expert_offsets, active_experts, num_active, W_gate, W_up, W_down, s_gate, s_up,
                           s_down, Y, stream=None) -> None:
    """moe_expert_ffn for callers that cannot allocate: no workspace argument; the library's
    fixed scratch area is used instead (see include/moe.h for its size limit and the rule
    that calls overlapping on one GPU race)."""
    P, H = xg.shape
    E, I, _ = W_gate.shape
    lib = load()
    f = lib.moe_expert_ffn_noalloc
    P_, i_ = ctypes.c_void_p, ctypes.c_int
    f.argtypes = [P_, P_, P_, P_, P_, P_, P_, P_, P_, P_, i_, i_, i_, i_, i_, P_, P_]
    f.restype = i_
    _check("moe_expert_ffn_noalloc", f(
        _ptr(xg), _ptr(expert_offsets), _ptr(active_experts), _ptr(num_active), _ptr(W_gate), _ptr(W_up),
        _ptr(W_down), _ptr(s_gate), _ptr(s_up), _ptr(s_down), _wtype(W_gate), H, I, E, P, _ptr(Y), _stream(stream)))


def moe_expert_ffn_noalloc_status(stream=None) -> int:
    """The status word moe_expert_ffn_noalloc's scratch holds after the stream's work so far (0 = no
    kernel gave up a wait)."""
    lib = load()
    f = lib.moe_expert_ffn_noalloc_status
    f.argtypes = [ctypes.c_void_p, ctypes.c_void_p]
    f.restype = ctypes.c_int
    word = ctypes.c_int32(-1)
    _check("moe_expert_ffn_noalloc_status", f(ctypes.addressof(word), _stream(stream)))
    return int(word.value)


def moe_gqa_workspace_size(B: int, h_q: int, h_kv: int, d: int, L_cap: int) -> int:
    return int(load().moe_gqa_workspace_size(B, h_q, h_kv, d, L_cap))


def alloc_gqa_workspace(B, h_q, h_kv, d, L_cap, device="cuda") -> torch.Tensor:
    """A zero-filled workspace for moe_gqa_decode (it must start zeroed; calls keep it so)."""
    n = moe_gqa_workspace_size(B, h_q, h_kv, d, L_cap)
    if n == 0:
        raise ValueError("invalid or unsupported sizes for moe_gqa_workspace_size")
    return torch.zeros(n, dtype=torch.uint8, device=device)


def moe_gqa_decode(q, k_cache, v_cache, seq_lens, scale: float, out, workspace, stream=None) -> None:
    """q [B,h_q,d], k_cache/v_cache [B,h_kv,L_cap,d] bf16, seq_lens [B] int32, out [B,h_q,d] bf16."""
    B, h_q, d = q.shape
    _, h_kv, L_cap, _ = k_cache.shape
    _check("moe_gqa_decode", load().moe_gqa_decode(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(seq_lens), B, h_q, h_kv, d, L_cap, float(scale), _ptr(out),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)))


def moe_expert_ffn_residual(xg, expert_offsets, active_experts, num_active, W_gate, W_up, W_down, s_gate, s_up,
                            s_down, Wr_gate, Wr_up, sr_gate, sr_up, Y, workspace, stream=None) -> None:
    """moe_expert_ffn with residual-split INT8 gate/up (W^Q + W^R; see include/moe.h)."""
    P, H = xg.shape
    E, I, _ = W_gate.shape
    _check("moe_expert_ffn_residual", load().moe_expert_ffn_residual(
        _ptr(xg), _ptr(expert_offsets), _ptr(active_experts), _ptr(num_active), _ptr(W_gate), _ptr(W_up),
        _ptr(W_down), _ptr(s_gate), _ptr(s_up), _ptr(s_down), _ptr(Wr_gate), _ptr(Wr_up), _ptr(sr_gate),
        _ptr(sr_up), H, I, E, P, _ptr(Y), _ptr(workspace), workspace.numel() * workspace.element_size(),
        _stream(stream)))


def moe_ffn_forward_residual(x, logits, W_gate, W_up, W_down, s_gate, s_up, s_down, Wr_gate, Wr_up, sr_gate, sr_up,
                             top_k, out, workspace, stream=None) -> None:
    """moe_ffn_forward with residual-split INT8 gate/up (W^Q + W^R; see include/moe.h)."""
    T, H = x.shape
    E, I, _ = W_gate.shape
    _check("moe_ffn_forward_residual", load().moe_ffn_forward_residual(
        _ptr(x), _ptr(logits), _ptr(W_gate), _ptr(W_up), _ptr(W_down), _ptr(s_gate), _ptr(s_up), _ptr(s_down),
        _ptr(Wr_gate), _ptr(Wr_up), _ptr(sr_gate), _ptr(sr_up), T, H, I, E, top_k, _ptr(out), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))
