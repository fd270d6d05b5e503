"""The C-ABI library builds, loads and exports what include/*.h declares; host-side
argument checks reject bad calls before any CUDA work (no GPU needed)."""
import ctypes
import glob
import os
import re

import pytest

from routed_expert_ffn_softmax_gb300 import build as moe_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = sorted(glob.glob(os.path.join(ROOT, "include", "*.h")))

OK, INVALID, UNSUPPORTED, WORKSPACE = 0, 1, 2, 3
BF16, INT8 = 0, 1


@pytest.fixture(scope="module")
def lib():
    path = moe_build.build()
    L = ctypes.CDLL(path)
    P, i, z = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    L.moe_workspace_size.argtypes = [i, i, i, i, i, i]
    L.moe_workspace_size.restype = z
    L.moe_status_string.argtypes = [i]
    L.moe_status_string.restype = ctypes.c_char_p
    L.moe_ffn_forward.argtypes = [P, P, P, P, P, P, P, P, i, i, i, i, i, i, P, P, z, P]
    L.moe_expert_ffn.argtypes = [P, P, P, P, P, P, P, P, P, P, i, i, i, i, i, P, P, z, P]
    L.moe_route_topk.argtypes = [P, i, i, i, P, P, P, P, P, P, P, P, P]
    L.moe_gather.argtypes = [P, i, i, i, P, P, P]
    L.moe_combine.argtypes = [P, P, P, i, i, i, P, P]
    L.moe_gqa_workspace_size.argtypes = [i, i, i, i, i]
    L.moe_gqa_workspace_size.restype = z
    L.moe_gqa_decode.argtypes = [P, P, P, P, i, i, i, i, i, ctypes.c_float, P, P, z, P]
    return L


def declared_functions():
    names = set()
    for h in HEADERS:
        src = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        names |= set(re.findall(r"\b(moe_[a-z_0-9]+)\s*\(", src))
    return sorted(names)


def test_header_declares_the_boundary():
    assert declared_functions() == sorted([
        "moe_status_string", "moe_workspace_size", "moe_route_topk", "moe_gather",
        "moe_expert_ffn", "moe_expert_ffn_noalloc", "moe_expert_ffn_noalloc_status", "moe_combine", "moe_ffn_forward",
        "moe_gqa_workspace_size", "moe_gqa_decode", "moe_expert_ffn_residual", "moe_ffn_forward_residual",
        "moe_set_decode_step_policy", "moe_ffn_forward_launches", "moe_test_expire_grid_barrier",
        "moe_set_expert_pass_tokens", "moe_test_expert_wait_limit"])


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_exports_are_c_symbols():
    out = os.popen(f"nm -D --defined-only {moe_build.LIB}").read()
    for name in declared_functions():
        assert re.search(rf"\bT {name}$", out, flags=re.M), name


def test_status_strings(lib):
    for code in range(5):
        s = lib.moe_status_string(code).decode()
        assert s.startswith("MOE_")
    assert b"unknown" in lib.moe_status_string(99)


def test_workspace_size(lib):
    ws = lib.moe_workspace_size
    n1 = ws(1, 4096, 14336, 8, 2, BF16)
    n64 = ws(64, 4096, 14336, 8, 2, BF16)
    assert 0 < n1 < n64
    assert n1 % 256 == 0
    # grows with the token block: xg (2 B) + Y (4 B) + h (2 B/I) per assignment
    assert n64 - n1 >= 63 * 2 * (2 * 4096 + 4 * 4096 + 2 * 14336)
    assert ws(0, 256, 512, 8, 2, BF16) > 0
    assert ws(-1, 256, 512, 8, 2, BF16) == 0
    assert ws(1, 256, 512, 8, 9, BF16) == 0          # top_k > E
    assert ws(1, 256, 512, 300, 2, BF16) == 0        # E > 256
    assert ws(1, 260, 512, 8, 2, BF16) == 0          # H % 8
    assert ws(1, 4096, 1536, 128, 8, INT8) > 0
    assert ws(1, 4096 + 64, 1536, 128, 8, INT8) == 0  # int8 needs H % 128 == 0
    assert ws(1, 256, 512, 8, 2, 7) == 0             # unknown weight type


FAKE = 1 << 20  # an aligned non-null address; never dereferenced (the calls below fail first)


def fwd(lib, T=1, H=256, I=512, E=8, k=2, wtype=BF16, x=FAKE, logits=FAKE, Wg=FAKE, Wu=FAKE, Wd=FAKE,
        sg=None, su=None, sd=None, out=FAKE, ws=FAKE, ws_bytes=None):
    if ws_bytes is None:
        ws_bytes = lib.moe_workspace_size(max(T, 0), H, I, E, k, wtype) if T >= 0 else 0
    return lib.moe_ffn_forward(x, logits, Wg, Wu, Wd, sg, su, sd, wtype, T, H, I, E, k, out, ws, ws_bytes, None)


def test_forward_rejects_bad_arguments_before_launch(lib):
    assert fwd(lib, T=-1) == INVALID
    assert fwd(lib, k=0) == INVALID
    assert fwd(lib, k=9) == INVALID
    assert fwd(lib, E=300, k=2) == UNSUPPORTED
    assert fwd(lib, H=260) == INVALID
    assert fwd(lib, I=0) == INVALID
    assert fwd(lib, wtype=5) == INVALID
    assert fwd(lib, x=None) == INVALID
    assert fwd(lib, Wd=None) == INVALID
    assert fwd(lib, x=FAKE + 8) == INVALID                 # x must be 16-byte aligned
    assert fwd(lib, ws=FAKE + 16) == INVALID               # workspace must be 256-byte aligned
    assert fwd(lib, ws_bytes=1024) == WORKSPACE
    # INT8: scales are required and dimensions must be multiples of 128
    assert fwd(lib, H=4096, I=1536, E=128, k=8, wtype=INT8) == INVALID
    assert fwd(lib, H=4096 + 8, I=1536, E=128, k=8, wtype=INT8, sg=FAKE, su=FAKE, sd=FAKE) == INVALID
    assert fwd(lib, H=4096, I=1536, E=128, k=8, wtype=INT8, sg=FAKE, su=FAKE, sd=FAKE, ws_bytes=16) == WORKSPACE
    # T = 0 is a no-op that touches nothing
    assert fwd(lib, T=0, x=None, logits=None, out=None, ws=None) in (OK, INVALID)
    assert fwd(lib, T=0) == OK


def test_other_entry_points_reject_bad_arguments(lib):
    F = FAKE
    assert lib.moe_route_topk(F, -1, 8, 2, F, F, F, F, F, F, F, F, None) == INVALID
    assert lib.moe_route_topk(F, 4, 8, 9, F, F, F, F, F, F, F, F, None) == INVALID
    assert lib.moe_route_topk(F, 4, 512, 2, F, F, F, F, F, F, F, F, None) == UNSUPPORTED
    assert lib.moe_route_topk(None, 4, 8, 2, F, F, F, F, F, F, F, F, None) == INVALID
    assert lib.moe_route_topk(F, 0, 8, 2, F, F, F, F, F, F, F, F, None) == OK
    assert lib.moe_gather(F, 4, 100, 2, F, F, None) == INVALID      # H % 8
    assert lib.moe_gather(F + 4, 4, 128, 2, F, F, None) == INVALID  # alignment
    assert lib.moe_gather(F, 0, 128, 2, F, F, None) == OK
    assert lib.moe_combine(F, F, F, 4, 0, 128, F, None) == INVALID
    assert lib.moe_combine(F, F, None, 4, 2, 128, F, None) == INVALID
    assert lib.moe_combine(F, F, F, 0, 2, 128, F, None) == OK
    ws_need = lib.moe_workspace_size(4, 256, 512, 8, 2, BF16)
    assert lib.moe_expert_ffn(F, F, F, F, F, F, F, None, None, None, BF16, 256, 512, 8, 8, F, F, 64, None) == WORKSPACE
    assert lib.moe_expert_ffn(F, F, F, F, F, F, F, None, None, None, BF16, 256, 512, 8, -1, F, F, ws_need, None) == INVALID
    assert lib.moe_expert_ffn(F, F, F, F, F, F, F, None, None, None, BF16, 256, 512, 8, 0, F, F, ws_need, None) == OK
    assert lib.moe_expert_ffn(F, F, F, F, F, F, F, None, None, None, INT8, 256, 512, 8, 8, F, F, ws_need, None) == INVALID


def test_gqa_workspace_size(lib):
    ws = lib.moe_gqa_workspace_size
    n = ws(64, 32, 4, 128, 8192)
    assert n > 0 and n % 256 == 0
    assert ws(2048, 64, 4, 128, 32768) == n           # independent of the sizes
    assert ws(1, 32, 3, 128, 16) == 0                 # h_q not a multiple of h_kv
    assert ws(1, 32, 1, 128, 16) == 0                 # group of 32 > 16
    assert ws(1, 32, 4, 64, 16) == 0                  # head dim other than 128
    assert ws(2049, 32, 4, 128, 16) == 0              # more sequences than supported
    assert ws(1, 32, 4, 128, 0) == 0                  # empty cache
    assert ws(-1, 32, 4, 128, 16) == 0


def gqa(lib, B=2, h_q=32, h_kv=4, d=128, L=256, scale=0.088, q=FAKE, k=FAKE, v=FAKE, lens=FAKE, out=FAKE, ws=FAKE,
        ws_bytes=None):
    if ws_bytes is None:
        ws_bytes = lib.moe_gqa_workspace_size(2, 32, 4, 128, 256)
    return lib.moe_gqa_decode(q, k, v, lens, B, h_q, h_kv, d, L, scale, out, ws, ws_bytes, None)


def test_gqa_rejects_bad_arguments_before_launch(lib):
    assert gqa(lib, B=-1) == INVALID
    assert gqa(lib, h_kv=3) == INVALID
    assert gqa(lib, h_q=64, h_kv=2) == UNSUPPORTED     # G = 32
    assert gqa(lib, d=64) == UNSUPPORTED
    assert gqa(lib, B=5000) == UNSUPPORTED
    assert gqa(lib, L=0) == INVALID
    assert gqa(lib, scale=float("inf")) == INVALID
    assert gqa(lib, scale=float("nan")) == INVALID
    assert gqa(lib, q=None) == INVALID
    assert gqa(lib, lens=None) == INVALID
    assert gqa(lib, k=FAKE + 8) == INVALID             # caches must be 16-byte aligned
    assert gqa(lib, lens=FAKE + 2) == INVALID
    assert gqa(lib, ws=FAKE + 16) == INVALID
    assert gqa(lib, ws_bytes=4096) == WORKSPACE
    assert gqa(lib, B=0, q=None, k=None, v=None, lens=None, out=None, ws=None) == OK


def test_gqa_tile_count_bound(lib):
    # 2048 sequences x 64 key/value heads x 2^17 tiles of 128 rows overflows the 32-bit tile count
    assert lib.moe_gqa_workspace_size(2048, 64, 64, 128, 1 << 24) == 0
    assert lib.moe_gqa_workspace_size(2048, 64, 64, 128, 1 << 20) > 0


def test_residual_entry_points_reject_bad_arguments(lib):
    F = FAKE
    P_, i, z = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    lib.moe_ffn_forward_residual.argtypes = [P_] * 12 + [i, i, i, i, i, P_, P_, z, P_]
    lib.moe_expert_ffn_residual.argtypes = [P_] * 14 + [i, i, i, i, P_, P_, z, P_]
    ws = lib.moe_workspace_size(4, 256, 256, 8, 2, INT8)
    f = lambda **kw: lib.moe_ffn_forward_residual(*[kw.get(n, F) for n in (
        "x", "lg", "Wg", "Wu", "Wd", "sg", "su", "sd", "rg", "ru", "srg", "sru")], kw.get("T", 4), kw.get("H", 256),
        256, 8, 2, F, F, kw.get("ws", ws), None)
    assert f(rg=None) == INVALID
    assert f(sru=None) == INVALID
    assert f(ru=F + 8) == INVALID          # residual parts must be 16-byte aligned
    assert f(H=264) == INVALID             # INT8 needs H % 128 == 0
    assert f(ws=64) == WORKSPACE
    assert f(T=0, rg=None) == OK           # T = 0 is a no-op
    assert lib.moe_expert_ffn_residual(*([F] * 10), None, F, F, F, 256, 256, 8, 8, F, F, ws, None) == INVALID


def test_decode_step_policy_and_launch_count(lib):
    """By batch shape the one-launch decode step runs for INT8 weights with at most one assignment per two experts
    and for BF16 weights up to two tokens (when the sizes allow it: T <= 32, P <= 256, H <= 16384, I <= 32768, H and
    I multiples of 128, INT8 of 512); the policy forces either path; host-only queries."""
    lib.moe_set_decode_step_policy.argtypes = [ctypes.c_int]
    lib.moe_set_decode_step_policy.restype = ctypes.c_int
    f = lib.moe_ffn_forward_launches
    f.argtypes = [ctypes.c_int] * 6
    f.restype = ctypes.c_int
    try:
        assert lib.moe_set_decode_step_policy(0) == OK
        assert f(64, 7168, 2048, 256, 8, BF16) == 5         # staged: route, gather, gate+up, down, combine
        assert f(512, 7168, 2048, 256, 8, BF16) == 6        # routing in two launches above 64 tokens
        assert f(64, 4096, 1536, 128, 8, INT8) == 6         # staged INT8: + the fp16 copy of h
        assert f(1, 4096, 1536, 128, 8, INT8) == 1          # INT8 at one token: the one-launch step
        assert f(8, 4096, 1536, 128, 8, INT8) == 1          # 64 assignments over 128 experts
        assert f(9, 4096, 1536, 128, 8, INT8) == 6          # 72: the separate launches
        assert f(3, 512, 512, 8, 2, INT8) == 6              # 6 assignments over 8 experts
        assert f(1, 7168, 2048, 256, 8, BF16) == 1          # BF16 at one and two tokens: the one-launch step
        assert f(2, 4096, 14336, 8, 2, BF16) == 1
        assert f(3, 4096, 14336, 8, 2, BF16) == 5           # three tokens: the separate launches
        assert f(16, 4096, 14336, 8, 2, BF16) == 5          # Mixtral-8x7B, 4 tokens per expert
        assert f(0, 256, 512, 8, 2, BF16) == 0
        assert f(1, 256, 512, 8, 9, BF16) == -1
        assert lib.moe_set_decode_step_policy(1) == OK
        assert f(1, 7168, 2048, 256, 8, BF16) == 5
        assert lib.moe_set_decode_step_policy(2) == OK
        assert f(1, 7168, 2048, 256, 8, BF16) == 1          # DeepSeek-V3, one token
        assert f(1, 4096, 1536, 128, 8, INT8) == 1          # Qwen3-235B INT8
        assert f(16, 4096, 14336, 8, 2, BF16) == 1
        assert f(1, 264, 200, 8, 2, BF16) == 5              # H, I not multiples of 128
        assert f(4, 384, 256, 8, 2, INT8) == 6              # INT8 with H not a multiple of 512
        assert f(33, 4096, 14336, 8, 2, BF16) == 5          # more than 32 tokens
        assert f(1, 16512, 1536, 128, 8, BF16) == 5         # H above 16384
        assert lib.moe_set_decode_step_policy(3) == INVALID
    finally:
        lib.moe_set_decode_step_policy(0)


def test_pass_tokens_size_the_workspace(lib):
    """BF16 workspaces hold stream-K partial slots for the pass size the batch shape picks (mean tokens per
    expert <= 40: 64, <= 96: 128, else 192 or 256 by the estimated largest expert) or the one forced;
    INT8 ones stay at 64-token slots."""
    ws = lib.moe_workspace_size
    f = lib.moe_set_expert_pass_tokens
    f.argtypes = [ctypes.c_int, ctypes.c_int]
    f.restype = ctypes.c_int
    slot64 = 4 * 256 * 2 * 16384                # 256 CTAs x 2 slots x (128 rows x 128 columns) fp32
    mix = lambda T, wt=BF16: ws(T, 4096, 14336, 8, 2, wt)   # mean tokens per expert = T / 4
    auto = {T: mix(T) for T in (64, 256, 1024, 4096)}
    int8 = mix(1024, INT8)
    try:
        assert f(64, 64) == OK
        base = {T: mix(T) for T in (64, 256, 1024, 4096)}
        assert mix(1024, INT8) == int8
        assert f(256, 64) == OK                  # gate+up at 256: slots of 128 x 512 columns
        assert mix(64) == base[64] + 3 * slot64
        assert f(64, 256) == OK                  # down at 256 on pairs: two tiles, 128 x 512 columns
        assert mix(64) == base[64] + 3 * slot64
        assert f(128, 0) == OK                   # gate+up at 128: 128 x 256; down by shape (64)
        assert mix(64) == base[64] + slot64
        assert f(192, 192) == OK                 # gate+up at 192: 128 x 384 columns
        assert mix(64) == base[64] + 2 * slot64
        assert f(96, 0) == INVALID and f(0, 32) == INVALID
    finally:
        assert f(0, 0) == OK
    assert auto[64] == base[64]                  # 16 per expert: 64-token passes
    assert auto[256] == base[256] + slot64       # 64 per expert: 128
    assert auto[1024] == base[1024] + 2 * slot64  # 256 per expert: 192 (the largest expert needs 2 ranks either way)
    assert auto[4096] == base[4096] + 3 * slot64  # 1024 per expert: 256 (at 192 it would need a sixth rank)
    assert mix(1024) == auto[1024]


def test_expert_wait_limit_hook_arguments(lib):
    f = lib.moe_test_expert_wait_limit
    f.argtypes = [ctypes.c_uint64]
    f.restype = ctypes.c_int
    try:
        assert f(50) == INVALID                # below 100 ns
        assert f(3 * 10**9) == INVALID         # above the normal 2 s limit
        assert f(1000) == OK
    finally:
        assert f(0) == OK


def test_grid_barrier_test_hook_arguments(lib):
    f = lib.moe_test_expire_grid_barrier
    f.argtypes = [ctypes.c_int, ctypes.c_uint64]
    f.restype = ctypes.c_int
    try:
        assert f(2, 10**6) == INVALID
        assert f(1, 10) == INVALID             # below 1 us
        assert f(1, 3 * 10**9) == INVALID      # above the normal 2 s limit
        assert f(1, 10**6) == OK
    finally:
        assert f(0, 0) == OK
