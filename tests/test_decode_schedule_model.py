"""Host model of the one-launch decode step's work split (csrc/decode_step.cu): the per-CTA tile
ranges of both phases, which CTA holds the head of every unit split between CTAs, and which later
pieces each head gathers. The kernel's waits on other CTAs end only if every later piece a head
waits for is published by the CTA the head expects, once per phase; these are checked here, with
the kernel's arithmetic restated in Python (the 32-bit forms next to the exact ones). No GPU.

The model follows the kernel: passes of kNE tokens per active expert in ascending expert order
(kNE = 1 at one token, 4 for INT8, 4 or 8 for BF16); a tile of a pass with n tokens costs
max(10, 4 + 3n) (BF16) or max(10, 4 + 5n) (INT8); gate+up tiles are pass-major with KIg = H / kKt
reduction tiles per (pass, 128-row block) unit; down tiles are row-block-major with KId = I / (2 kKt);
CTA c's range starts at the first tile whose cost position is at least floor(c * C / N_used)."""
import numpy as np
import pytest


def tile_cost(n, int8):
    return max(10, 4 + (5 if int8 else 3) * n)


def tokens_per_pass(T, E, k, int8):
    if T == 1:
        return 1
    if int8:
        return 4
    return 4 if T * k <= E else 8


def scaled32(c, C, N):
    """floor(c * C / N) as the kernel computes it in 32-bit arithmetic."""
    q, r = C // N, C % N
    assert c * r < 2 ** 31 and c * q < 2 ** 31
    return c * q + (c * r) // N


def cta_at32(pos, C, N):
    """The kernel's cta_at: an fp32 estimate, then exact steps."""
    c = int(np.float32(np.float32(pos) * np.float32(N)) / np.float32(C))
    c = max(0, min(N - 1, c))
    while c + 1 < N and scaled32(c + 1, C, N) <= pos:
        c += 1
    while c > 0 and scaled32(c, C, N) > pos:
        c -= 1
    return c


def schedule(counts, H, I, int8, kNE, N=152):
    kKt = 128 if int8 else 64
    passes = [min(kNE, c - j) for c in counts for j in range(0, c, kNE)]
    NU = len(passes)
    qc = [tile_cost(n, int8) for n in passes]
    pc = np.concatenate([[0], np.cumsum(qc)]).astype(np.int64)
    RBg, KIg = I // 128, H // kKt
    RBd, KId = H // 128, I // (2 * kKt)
    TPg = RBg * KIg
    Wg, Wd = NU * TPg, NU * RBd * KId
    PC = int(pc[NU])
    Cg, Rd = PC * TPg, PC * KId
    Cd = Rd * RBd
    kmax = tile_cost(kNE, int8)
    Ng, Nd = min(N, max(1, Cg // kmax)), min(N, max(1, Cd // kmax))

    def pass_at(X):
        return int(np.searchsorted(pc[:NU], X, side="right") - 1)

    def pos_gu(i):
        q = i // TPg
        return int(pc[q]) * TPg + (i - q * TPg) * qc[q]

    def first_gu(X):
        if X >= Cg:
            return Wg
        q = pass_at(X // TPg)
        return q * TPg + (X - int(pc[q]) * TPg + qc[q] - 1) // qc[q]

    def pos_dn(i):
        u = i // KId
        rb, q = u // NU, u % NU
        return rb * Rd + int(pc[q]) * KId + (i - u * KId) * qc[q]

    def first_dn(X):
        if X >= Cd:
            return Wd
        rb, rem = X // Rd, X % Rd
        q = pass_at(rem // KId)
        return (rb * NU + q) * KId + (rem - int(pc[q]) * KId + qc[q] - 1) // qc[q]

    phases = {"gate+up": (Ng, Cg, Wg, KIg, first_gu, pos_gu), "down": (Nd, Cd, Wd, KId, first_dn, pos_dn)}
    return dict(NU=NU, Cg=Cg, Cd=Cd, Wg=Wg, Wd=Wd, phases=phases)


def check(counts, H, I, int8, kNE, N=152):
    s = schedule(counts, H, I, int8, kNE, N)
    assert s["Cg"] < 2 ** 31 and s["Cd"] < 2 ** 31 and s["Wg"] < 2 ** 31 and s["Wd"] < 2 ** 31
    for phase, (Nx, Cx, Wx, KI, first, pos) in s["phases"].items():
        # the ranges: [first(scaled(c)), first(scaled(c + 1))) for the CTAs taking part, empty above
        rng = [(first(scaled32(c, Cx, Nx)), first(scaled32(c + 1, Cx, Nx))) if c < Nx else (Wx, Wx)
               for c in range(N)]
        for c in range(Nx):
            assert scaled32(c, Cx, Nx) == c * Cx // Nx
        assert rng[0][0] == 0 and rng[Nx - 1][1] == Wx, phase
        for c in range(1, Nx):
            assert rng[c][0] == rng[c - 1][1], (phase, c)          # every tile once, in order
        assert all(b < e for b, e in rng[:Nx]), phase              # every CTA taking part holds a tile
        later, heads = {}, {}
        for c, (b, e) in enumerate(rng):
            i = b
            while i < e:
                u = i // KI
                ub, ue = u * KI, u * KI + KI
                if ub < b:                                          # a later piece: the range's first unit
                    assert i == b and c not in later, (phase, c)
                    later[c] = u
                elif ue > e:                                        # the head: the range's last unit
                    heads[c] = (u, ue)
                i = min(ue, e)
        for c, (u, ue) in heads.items():
            c_last = cta_at32(pos(ue - 1), Cx, Nx)
            assert c_last == ((pos(ue - 1) + 1) * Nx - 1) // Cx
            assert c_last > c
            for c2 in range(c + 1, c_last + 1):                     # the flags the head waits for
                assert later.get(c2) == u, (phase, c, c2)
        for c2, u in later.items():                                 # every later piece has a head
            h = cta_at32(pos(u * KI), Cx, Nx)
            assert heads.get(h, (None,))[0] == u, (phase, c2)
    return s


def seeded_counts(seed, T, E, k, skew=()):
    """Per-expert token counts of T tokens routed to k distinct experts each (uniform, or with the
    skewed experts in every token's choice)."""
    rng = np.random.default_rng(seed)
    counts = np.zeros(E, int)
    for _ in range(T):
        chosen = list(skew[:k]) + list(rng.choice([e for e in range(E) if e not in skew], k - len(skew[:k]), replace=False))
        counts[chosen] += 1
    return [int(c) for c in counts if c > 0]


# the shapes of tests/test_decode_step.py and the bench's decode workloads
CASES = [
    (1, 256, 512, 8, 2, False, ()), (8, 256, 512, 8, 2, False, ()), (3, 384, 640, 16, 4, False, ()),
    (32, 512, 256, 64, 4, False, ()), (20, 256, 384, 8, 2, False, (0,)), (6, 128, 128, 4, 4, False, ()),
    (5, 1024, 256, 256, 8, False, ()), (1, 512, 512, 128, 8, True, ()), (8, 1024, 512, 128, 8, True, ()),
    (16, 512, 1024, 32, 2, True, (3,)), (32, 512, 512, 64, 8, True, ()), (2, 1536, 512, 8, 2, True, ()),
    (8, 512, 512, 64, 2, False, (0,)), (12, 512, 512, 64, 4, True, (1,)),
    (1, 4096, 1536, 128, 8, True, ()), (4, 4096, 1536, 128, 8, True, ()), (16, 4096, 1536, 128, 8, True, ()),
    (1, 4096, 14336, 8, 2, False, ()), (4, 4096, 14336, 8, 2, False, ()), (16, 4096, 14336, 8, 2, False, ()),
    (1, 7168, 2048, 256, 8, False, ()), (4, 7168, 2048, 256, 8, False, ()), (32, 7168, 2048, 256, 8, False, ()),
    (1, 6144, 16384, 8, 2, False, ()), (4, 6144, 16384, 8, 2, False, (0, 1)),
]


@pytest.mark.parametrize("T,H,I,E,k,int8,skew", CASES)
def test_heads_wait_only_for_pieces_that_are_published(T, H, I, E, k, int8, skew):
    for seed in range(3):
        check(seeded_counts(seed, T, E, k, skew), H, I, int8, tokens_per_pass(T, E, k, int8))


def test_fewer_ctas_than_sms():
    """Launches capped below one CTA per SM (max_ctas) keep the same properties."""
    for N in (1, 2, 7, 33, 100):
        check(seeded_counts(5, 4, 128, 8), 4096, 1536, True, 4, N=N)
        check(seeded_counts(6, 3, 16, 4), 384, 640, False, 4, N=N)


def test_largest_sizes_stay_32_bit():
    """The decode step's limits (T * k <= 256, H <= 16384, I <= 32768): the total cost is largest for
    256 single-token passes (a pass of n tokens costs at most 10 per token at n = 1); every cost
    position and product stays below 2^31 there and for full passes."""
    for int8 in (False, True):
        kNE = 4 if int8 else 8
        for counts in ([1] * 256, [kNE] * (256 // kNE)):        # 256 assignments
            s = schedule(counts, 16384, 32768, int8, kNE)
            assert s["Cg"] < 2 ** 31 and s["Cd"] < 2 ** 31 and s["Wg"] < 2 ** 31 and s["Wd"] < 2 ** 31
            for c in range(153):
                scaled32(c, s["Cg"], 152)
                scaled32(c, s["Cd"], 152)


def test_fp32_estimate_of_the_cta_is_exact():
    rng = np.random.default_rng(11)
    for _ in range(5000):
        N = int(rng.integers(1, 153))
        C = int(rng.integers(N, 2 ** 31 - 1))
        for pos in (0, C - 1, int(rng.integers(0, C))):
            assert cta_at32(pos, C, N) == ((pos + 1) * N - 1) // C
