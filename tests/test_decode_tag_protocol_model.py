"""Random-interleaving model of the one-launch decode step's hand-off of split units
(csrc/decode_step.cu): later pieces store (tag, value) pairs into their CTA's partial slot, each
head's helper gathers the later pieces of its unit once they carry the phase's tag, and a grid
barrier separates gate+up from down. No GPU: CTAs and helpers are coroutines over a shared memory,
run in random orders over consecutive launches on one workspace; every value a head accepts must
be the one its unit's later piece wrote in this launch and phase.

What the model keeps from the kernel: the tag is 2 * (release word at entry) + 1 for gate+up and
+ 2 for down, the release word advancing once per launch when the last CTA arrives; a CTA's compute
posts a head's gather when it begins the head unit (the helper runs it meanwhile) and needs the
gathered sum at the unit's end; a down unit's tiles need h, i.e. the barrier open, while a down
head's gather may begin before (its first unit can be the head); a CTA arrives at the barrier after
its gate+up head has its sum. Two altered tag rules, one per launch only and one without the
launch, must fail: the model sees the faults the tags exist to prevent."""
import random

import pytest

from test_decode_schedule_model import schedule, scaled32, cta_at32, seeded_counts, tokens_per_pass


def ranges_and_roles(s, N):
    """Per phase: each CTA's units in range order with their role, and each head's later CTAs."""
    out = {}
    for phase, (Nx, Cx, Wx, KI, first, pos) in s["phases"].items():
        per_cta = []
        for c in range(N):
            b, e = (first(scaled32(c, Cx, Nx)), first(scaled32(c + 1, Cx, Nx))) if c < Nx else (Wx, Wx)
            units, i = [], b
            while i < e:
                u = i // KI
                ub, ue = u * KI, u * KI + KI
                if ub < b:
                    units.append((u, "piece", ()))
                elif ue > e:
                    c_last = cta_at32(pos(ue - 1), Cx, Nx)
                    units.append((u, "head", tuple(range(c + 1, c_last + 1))))
                else:
                    units.append((u, "whole", ()))
                i = min(ue, e)
            per_cta.append(units)
        out[phase] = per_cta
    return out


class Deadlock(Exception):
    pass


def run_launches(roles_per_launch, N, seed, tag_rule):
    """Run consecutive steps (one routing each) on one memory in a random interleaving; returns the
    number of accepted gathers. tag_rule(release_word, phase_index) gives the phase's tag."""
    rng = random.Random(seed)
    mem = {"slot": [(0, None)] * N, "arrived": 0, "release": 0}
    accepted = 0
    for launch, roles in enumerate(roles_per_launch):
        procs = []

        def gather(c, phase, ph, unit, later, tag, done):
            nonlocal accepted
            for c2 in later:
                yield lambda c2=c2: mem["slot"][c2][0] == tag
                got = mem["slot"][c2][1]
                assert got == (launch, phase, unit), f"head {c} of {phase} unit {unit} took {got} from CTA {c2}"
                accepted += 1
            done.append(True)

        def cta(c):
            entry = mem["release"]  # read at entry; no CTA can advance it before every CTA has arrived
            for ph, phase in enumerate(("gate+up", "down")):
                tag = tag_rule(entry, ph)
                if phase == "down":
                    opened = lambda: mem["release"] != entry
                for (u, role, later) in roles[phase][c]:
                    done = []
                    if role == "head":  # posted when the unit begins; the helper gathers meanwhile
                        procs.append(gather(c, phase, ph, u, later, tag, done))
                    if phase == "down":
                        yield opened  # the unit's tiles need h
                    yield None  # the unit's tiles
                    if role == "piece":
                        mem["slot"][c] = (tag, (launch, phase, u))
                    elif role == "head":
                        yield lambda done=done: bool(done)  # the gathered sum, at the unit's end
                if phase == "gate+up":  # arrive: the last arriver resets the count and releases
                    mem["arrived"] += 1
                    if mem["arrived"] == N:
                        mem["arrived"] = 0
                        mem["release"] += 1
            yield None

        procs.extend(cta(c) for c in range(N))
        waits = {id(p): None for p in procs}
        live = list(procs)
        while live:
            runnable = [p for p in live if waits[id(p)] is None or waits[id(p)]()]
            if not runnable:
                raise Deadlock(f"launch {launch}: {len(live)} coroutines wait forever")
            p = rng.choice(runnable)
            try:
                waits[id(p)] = next(p)
            except StopIteration:
                live.remove(p)
            for q in procs:  # coroutines spawned meanwhile
                if id(q) not in waits:
                    waits[id(q)] = None
                    live.append(q)
    return accepted


def adopted(release_word, phase_index):
    return 2 * release_word + 1 + phase_index


CASES = [  # (T, H, I, E, k, int8, N): short ranges, units spanning up to four CTAs
    (3, 384, 640, 16, 4, False, 12),
    (1, 512, 512, 128, 8, True, 29),
    (2, 256, 512, 8, 2, False, 9),
]


def launches_for(T, H, I, E, k, int8, N, n_launches, seed):
    """Each launch routes its own tokens (seeded), so its pieces and heads differ from the last's."""
    out = []
    for L in range(n_launches):
        s = schedule(seeded_counts(seed * 7 + L, T, E, k), H, I, int8, tokens_per_pass(T, E, k, int8), N)
        out.append(ranges_and_roles(s, N))
    return out


@pytest.mark.parametrize("T,H,I,E,k,int8,N", CASES)
def test_heads_accept_only_this_launch_and_phase(T, H, I, E, k, int8, N):
    accepted = 0
    for seed in range(30):
        runs = launches_for(T, H, I, E, k, int8, N, 3, seed)
        accepted += run_launches(runs, N, seed, adopted)
    assert accepted > 0  # heads gathered later pieces


def faults_under(tag_rule, n_launches):
    faults = 0
    for seed in range(30):
        try:
            run_launches(launches_for(3, 384, 640, 16, 4, False, 12, n_launches, seed), 12, seed, tag_rule)
        except (AssertionError, Deadlock):
            faults += 1
    return faults


def test_one_tag_per_launch_for_both_phases_fails():
    """With the down phase sharing gate+up's tag, a down head that gathers before the barrier can
    take a later CTA's gate+up sum (the fault the two per-phase tags prevent)."""
    assert faults_under(lambda e, ph: e + 1, 2) > 0


def test_tags_without_the_launch_fail():
    """With the same tags every launch, a head can take the previous launch's sum."""
    assert faults_under(lambda e, ph: 1 + ph, 3) > 0
