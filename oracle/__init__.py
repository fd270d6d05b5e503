"""ctypes front end of the plain CPU oracle (oracle/moe_oracle.cpp, oracle/gqa_oracle.cpp).

TEST INFRASTRUCTURE ONLY: tests/, __graft_entry__.smoke() and bench.py's
CPU-baseline leg may import this package; the CUDA product path never does.

Arrays are numpy or CPU torch tensors. bf16 tensors travel as their raw
uint16 bit patterns. Every function here only marshals arguments; the
arithmetic is in the two C++ files.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRCS = [os.path.join(_HERE, "moe_oracle.cpp"), os.path.join(_HERE, "gqa_oracle.cpp")]
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

WTYPE = {"bf16": 0, "int8": 1}


def build(force: bool = False) -> str:
    """Compile liboracle.so with g++ (sequential fp32 sums: -ffp-contract=off)."""
    if not force and os.path.exists(_LIB) and all(os.path.getmtime(_LIB) >= os.path.getmtime(f) for f in _SRCS):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["g++", "-O2", "-std=c++17", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", "-o", tmp, *_SRCS]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            P = ctypes.c_void_p
            i = ctypes.c_int
            lib.oracle_route.argtypes = [P, i, i, i, P, P, P, P, P, P, P, P]
            lib.oracle_route.restype = i
            lib.oracle_gateup_token.argtypes = [P, P, P, P, P, i, i, i, P, P, P]
            lib.oracle_gateup_token.restype = None
            lib.oracle_down_token.argtypes = [P, P, P, i, i, i, P]
            lib.oracle_down_token.restype = None
            lib.oracle_combine_token.argtypes = [P, P, i, i, P, P]
            lib.oracle_combine_token.restype = None
            lib.oracle_forward.argtypes = [P, P, P, P, P, P, P, P, i, i, i, i, i, i, P, P, P, P, P, P]
            lib.oracle_forward.restype = i
            lib.oracle_f32_to_bf16.argtypes = [P, ctypes.c_long, P]
            lib.oracle_f32_to_bf16.restype = None
            lib.oracle_gateup_token_residual.argtypes = [P] * 9 + [i, i, P, P, P]
            lib.oracle_gateup_token_residual.restype = None
            lib.oracle_forward_residual.argtypes = [P] * 12 + [i, i, i, i, i, P, P]
            lib.oracle_forward_residual.restype = i
            lib.oracle_gqa_decode.argtypes = [P, P, P, P, i, i, i, i, i, ctypes.c_float, P, P]
            lib.oracle_gqa_decode.restype = i
            lib.oracle_f64_to_bf16.argtypes = [P, ctypes.c_long, P]
            lib.oracle_f64_to_bf16.restype = None
            _lib = lib
    return _lib


def _np(a, dtype=None):
    """numpy view (C-contiguous) of a numpy array or CPU torch tensor; bf16 -> uint16 bits."""
    if a is None:
        return None
    try:
        import torch
        if isinstance(a, torch.Tensor):
            a = a.detach().cpu().contiguous()
            if a.dtype == torch.bfloat16:
                a = a.view(torch.int16).numpy().view(np.uint16)
            else:
                a = a.numpy()
    except ImportError:  # pragma: no cover
        pass
    a = np.ascontiguousarray(a)
    if dtype is not None and a.dtype != dtype:
        raise TypeError(f"expected {dtype}, got {a.dtype}")
    return a


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def route(logits, top_k: int):
    """Routing of logits [T,E] f32. Returns dict of numpy arrays (see moe_oracle.cpp)."""
    lg = _np(logits, np.float32)
    T, E = lg.shape
    P = T * top_k
    out = dict(
        ids=np.zeros((T, top_k), np.int32), w=np.zeros((T, top_k), np.float32),
        counts=np.zeros(E, np.int32), offsets=np.zeros(E + 1, np.int32),
        sorted_token=np.zeros(P, np.int32), inv_pos=np.zeros((T, top_k), np.int32),
        active=np.zeros(E, np.int32), num_active=np.zeros(1, np.int32),
    )
    rc = _load().oracle_route(_p(lg), T, E, top_k, *(_p(out[n]) for n in (
        "ids", "w", "counts", "offsets", "sorted_token", "inv_pos", "active", "num_active")))
    if rc != 0:
        raise ValueError("oracle_route: bad sizes")
    out["num_active"] = int(out["num_active"][0])
    out["active"] = out["active"][: out["num_active"]].copy()
    return out


def gateup_token(x_row, Wg_e, Wu_e, sg_e=None, su_e=None, wtype="bf16"):
    """One token through one expert's gate/up: returns (h bf16 bits [I], g f32 [I], u f32 [I])."""
    x = _np(x_row, np.uint16)
    wt = WTYPE[wtype]
    wg = _np(Wg_e, np.uint16 if wt == 0 else np.int8)
    wu = _np(Wu_e, np.uint16 if wt == 0 else np.int8)
    I, H = wg.shape
    assert x.shape == (H,) and wu.shape == (I, H)
    sg = _np(sg_e, np.float32) if wt else None
    su = _np(su_e, np.float32) if wt else None
    h = np.zeros(I, np.uint16)
    g = np.zeros(I, np.float32)
    u = np.zeros(I, np.float32)
    _load().oracle_gateup_token(_p(x), _p(wg), _p(wu), _p(sg), _p(su), wt, H, I, _p(h), _p(g), _p(u))
    return h, g, u


def down_token(h_row, Wd_e, sd_e=None, wtype="bf16"):
    """One token's intermediate through one expert's down projection: y f32 [H]."""
    h = _np(h_row, np.uint16)
    wt = WTYPE[wtype]
    wd = _np(Wd_e, np.uint16 if wt == 0 else np.int8)
    H, I = wd.shape
    assert h.shape == (I,)
    sd = _np(sd_e, np.float32) if wt else None
    y = np.zeros(H, np.float32)
    _load().oracle_down_token(_p(h), _p(wd), _p(sd), wt, H, I, _p(y))
    return y


def combine_token(y_slots, w_slots):
    """Combine of one token: y [k,H] f32, w [k] f32 -> (out bf16 bits [H], out f32 [H])."""
    y = _np(y_slots, np.float32)
    w = _np(w_slots, np.float32)
    k, H = y.shape
    out = np.zeros(H, np.uint16)
    of = np.zeros(H, np.float32)
    _load().oracle_combine_token(_p(y), _p(w), k, H, _p(out), _p(of))
    return out, of


def forward(x, logits, W_gate, W_up, W_down, s_gate=None, s_up=None, s_down=None,
            wtype="bf16", top_k=2, intermediates=False):
    """Whole routed-expert FFN. Returns dict(out bf16 bits [T,H], out_f32 [T,H], ...)."""
    xa = _np(x, np.uint16)
    lg = _np(logits, np.float32)
    wt = WTYPE[wtype]
    wdt = np.uint16 if wt == 0 else np.int8
    wg, wu, wd = _np(W_gate, wdt), _np(W_up, wdt), _np(W_down, wdt)
    T, H = xa.shape
    E, I, H2 = wg.shape
    assert H2 == H and lg.shape == (T, E) and wd.shape == (E, H, I)
    sg = _np(s_gate, np.float32) if wt else None
    su = _np(s_up, np.float32) if wt else None
    sd = _np(s_down, np.float32) if wt else None
    out = np.zeros((T, H), np.uint16)
    of = np.zeros((T, H), np.float32)
    res = dict(out=out, out_f32=of)
    ids = w = h = y = None
    if intermediates:
        ids = np.zeros((T, top_k), np.int32)
        w = np.zeros((T, top_k), np.float32)
        h = np.zeros((T, top_k, I), np.uint16)
        y = np.zeros((T, top_k, H), np.float32)
        res.update(ids=ids, w=w, h=h, y=y)
    rc = _load().oracle_forward(_p(xa), _p(lg), _p(wg), _p(wu), _p(wd), _p(sg), _p(su), _p(sd), wt,
                                T, H, I, E, top_k, _p(out), _p(of), _p(ids), _p(w), _p(h), _p(y))
    if rc != 0:
        raise ValueError("oracle_forward: bad sizes")
    return res


def gateup_token_residual(x_row, qQg, sQg, qRg, sRg, qQu, sQu, qRu, sRu):
    """Residual-split gate/up of one token through one expert ([I,H] int8 parts, [I,H/128] scales):
    returns (h bf16 bits [I], g f32 [I], u f32 [I])."""
    x = _np(x_row, np.uint16)
    parts = [_np(a, np.int8 if i % 2 == 0 else np.float32) for i, a in enumerate((qQg, sQg, qRg, sRg, qQu, sQu,
                                                                                 qRu, sRu))]
    I, H = parts[0].shape
    h = np.zeros(I, np.uint16)
    g = np.zeros(I, np.float32)
    u = np.zeros(I, np.float32)
    _load().oracle_gateup_token_residual(_p(x), *(_p(a) for a in parts), H, I, _p(h), _p(g), _p(u))
    return h, g, u


def forward_residual(x, logits, W_gate, s_gate, Wr_gate, sr_gate, W_up, s_up, Wr_up, sr_up, W_down, s_down,
                     top_k=8):
    """Routed-expert FFN with residual-split gate/up (see moe_oracle.cpp). Returns dict(out, out_f32)."""
    xa = _np(x, np.uint16)
    lg = _np(logits, np.float32)
    q = [_np(a, np.int8) for a in (W_gate, Wr_gate, W_up, Wr_up, W_down)]
    sc = [_np(a, np.float32) for a in (s_gate, sr_gate, s_up, sr_up, s_down)]
    T, H = xa.shape
    E, I, _ = q[0].shape
    out = np.zeros((T, H), np.uint16)
    of = np.zeros((T, H), np.float32)
    rc = _load().oracle_forward_residual(_p(xa), _p(lg), _p(q[0]), _p(sc[0]), _p(q[1]), _p(sc[1]), _p(q[2]),
                                         _p(sc[2]), _p(q[3]), _p(sc[3]), _p(q[4]), _p(sc[4]), T, H, I, E, top_k,
                                         _p(out), _p(of))
    if rc != 0:
        raise ValueError("oracle_forward_residual: bad sizes")
    return dict(out=out, out_f32=of)


def gqa_decode(q, k_cache, v_cache, seq_lens, scale: float):
    """Decode-phase GQA attention (gqa_oracle.cpp). q [B,h_q,d], K/V [B,h_kv,L_cap,d] bf16,
    seq_lens [B] int32. Returns dict(out bf16 bits [B,h_q,d], out_f64 [B,h_q,d])."""
    qa = _np(q, np.uint16)
    ka = _np(k_cache, np.uint16)
    va = _np(v_cache, np.uint16)
    ln = _np(seq_lens, np.int32)
    B, h_q, d = qa.shape
    B2, h_kv, L_cap, d2 = ka.shape
    assert B2 == B and d2 == d and va.shape == ka.shape and ln.shape == (B,)
    out = np.zeros((B, h_q, d), np.uint16)
    of = np.zeros((B, h_q, d), np.float64)
    rc = _load().oracle_gqa_decode(_p(qa), _p(ka), _p(va), _p(ln), B, h_q, h_kv, d, L_cap,
                                   float(scale), _p(out), _p(of))
    if rc != 0:
        raise ValueError("oracle_gqa_decode: bad sizes or sequence lengths")
    return dict(out=out, out_f64=of)


def f64_to_bf16_bits(a):
    a = _np(a, np.float64)
    out = np.zeros(a.shape, np.uint16)
    _load().oracle_f64_to_bf16(_p(a), a.size, _p(out))
    return out


def f32_to_bf16_bits(a):
    a = _np(a, np.float32)
    out = np.zeros(a.shape, np.uint16)
    _load().oracle_f32_to_bf16(_p(a), a.size, _p(out))
    return out


def bf16_bits_to_f32(b):
    """Widen bf16 bit patterns to fp32 (exact)."""
    b = np.ascontiguousarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)
