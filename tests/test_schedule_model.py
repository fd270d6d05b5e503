"""The BF16 expert kernels' work split, modelled on the host (no GPU): the same integer formulas as
csrc/expert_tc.cuh's schedule, checked over many shapes.

- Pieces: at passes of more than 64 tokens, whole units in waves over the columns (column c takes
  units c, c + NC, ...) and the last NC..2NC units split stream-K; at 64-token passes, stream-K over
  all units. Every (unit, stage) must be covered exactly once; a column holds at most two partial
  pieces, in distinct slots; the columns that hold a split unit's pieces are the ones the last
  arriver's reduction visits, each at the slot it reads.
- Rank shares: an expert's tokens in rounds of g * kN, each round split over the g ranks in shares of
  a multiple of 16 that fit a pass; every token belongs to exactly one rank's share.
"""
import random

import pytest


def pieces(U, KI, ncols, waves_allowed):
    waves = waves_allowed and U >= 2 * ncols
    NC = ncols if waves else min(U * KI, ncols)
    D = (U // NC - 1) * NC if waves else 0
    Wt = (U - D) * KI
    out = {}
    for col in range(ncols + 1):  # one column past the grid: idle
        nW = (U // NC - 1) if (waves and col < NC) else 0
        sb = col * Wt // NC if col < NC else 0
        se = (col + 1) * Wt // NC if col < NC else 0
        n_sk = (se - 1) // KI - sb // KI + 1 if sb < se else 0
        ps = []
        for p in range(nW + n_sk):
            if p < nW:
                ps.append((p * NC + col, 0, KI, None))
            else:
                uf = sb // KI
                ut = uf + (p - nW)
                kb = sb - uf * KI if p == nW else 0
                ke = min(KI, se - ut * KI)
                ps.append((D + ut, kb, ke, 0 if p == nW else 1))
        out[col] = ps
    return out, NC, D, Wt


def check_pieces(U, KI, ncols, waves_allowed):
    out, NC, D, Wt = pieces(U, KI, ncols, waves_allowed)
    cover, partial = {}, {}
    for col, ps in out.items():
        slots = [p[3] for p in ps if not (p[1] == 0 and p[2] == KI)]
        assert len(slots) == len(set(slots)) and len(slots) <= 2, (col, ps)
        for u, kb, ke, slot in ps:
            assert 0 <= kb < ke <= KI
            for k in range(kb, ke):
                assert (u, k) not in cover, (u, k)
                cover[(u, k)] = col
            if not (kb == 0 and ke == KI):
                partial.setdefault(u, []).append((col, slot))
    assert len(cover) == U * KI
    col_of = lambda i: ((i + 1) * NC - 1) // Wt
    for u, lst in partial.items():
        ut = u - D
        cf, cl = col_of(ut * KI), col_of(ut * KI + KI - 1)
        assert sorted(c for c, _ in lst) == list(range(cf, cl + 1)), (u, lst, cf, cl)
        for c, slot in lst:
            assert slot == (0 if ut == (c * Wt // NC) // KI else 1)


def rank_share(mr, g):
    return ((mr + g - 1) // g + 15) // 16 * 16


def check_shares(ntok, kN, g):
    span = g * kN
    rounds = (ntok + span - 1) // span
    seen = []
    for rnd in range(rounds):
        left = ntok - rnd * span
        mr = min(left, span)
        share = rank_share(mr, g)
        assert share % 16 == 0 and share <= kN
        for rank in range(g):
            off = rank * share
            n = max(0, min(mr - off, share))
            seen += list(range(rnd * span + off, rnd * span + off + n))
    assert seen == list(range(ntok))


@pytest.mark.parametrize("seed", range(4))
def test_piece_schedule_covers_every_stage_once(seed):
    rng = random.Random(seed)
    for _ in range(300):
        U, KI = rng.randint(1, 400), rng.randint(1, 64)
        ncols = rng.choice([152, 76, 50, 38, 25, 19, 7, 1])
        check_pieces(U, KI, ncols, waves_allowed=rng.random() < 0.5)
    for U, KI, ncols in [(448, 64, 25), (64, 224, 25), (128, 112, 152)]:
        check_pieces(U, KI, ncols, True)
        check_pieces(U, KI, ncols, False)


def test_rank_shares_cover_every_token_once():
    for ntok in list(range(1, 300)) + list(range(300, 2200, 53)):
        for kN in (64, 128, 192, 256):
            for g in range(1, 9):
                check_shares(ntok, kN, g)
