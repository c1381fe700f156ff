"""The mbarrier protocol of the persistent decode kernels, on the CPU.

An mbarrier keeps only the parity of its phase. A wait for the completion of
phase n (parity n % 2) passes whenever the barrier's count of completed
phases c has c % 2 != n % 2: at c = n + 1 as intended, but also at
c = n - 1, while phase n - 1 is still in progress. The kernels therefore
rely on two ownership rules, stated in their sources:

* state stages (stream and delta kernels): unit u goes to stage u mod NS and
  to consumer group u mod G, and NS is a multiple of G, so each stage serves
  one group only and that group waits for a stage's next fill only after
  consuming its previous one (the fused Mamba-2 step gives each group its
  own ring of NS / G stages outright, which is the same rule);
* vector slots of the delta kernel: prep warp w writes the slots of heads
  w, w + NP, ... (slot li mod NSL), consumer group g takes units
  g, g + G, ... (head = unit // nrb); NSL is a multiple of NP and NSL * nrb
  a multiple of G, so every fill of a slot comes from one warp, in order, and
  every group consumes every fill of each slot it uses. The tensor-core
  verify kernel's prep stages follow the same scheme: head li goes to warp
  li mod NP and to that warp's stage (li / NP) mod depth, that is, to slot
  li mod (NP * depth) of a warp's own, and its configurations keep
  NP * depth * nrb a multiple of G.

The fused Mamba-2 step's rings add two details: a fold unit takes FS
consecutive stages of its group's ring (the second one, past the ring's end,
waits for the flipped parity), and the launch requires at least FS stages
per group.

This file runs these protocols, wait for wait and arrival for arrival as the
kernels issue them, under many random interleavings (copies landing late,
warps running ahead), and checks that nobody reads a fill meant for another
unit or head, that no fill overwrites data still being read and that nothing
deadlocks. A mutant of each rule (11 stages for 4 groups; slot counts that
break either multiple; a ring shorter than a fold unit; no parity flip for a
fold unit's wrapped second stage) must fail the same check.
"""

import random

import pytest


class Barrier:
    """Completed-phase count of one mbarrier with `count` arrivals per phase."""

    def __init__(self, count=1):
        self.count, self.pending, self.c = count, count, 0

    def passes(self, parity):
        return self.c % 2 != parity

    def arrive(self):
        self.pending -= 1
        if self.pending == 0:
            self.c += 1
            self.pending = self.count


def run_stages(NS, G, U, seed):
    """Producer, copies in flight and G consumer groups over U units; returns
    the violations seen (reads of another unit's fill, overwrites of a fill
    not yet released)."""
    rng = random.Random(seed)
    full = [Barrier() for _ in range(NS)]
    empty = [Barrier() for _ in range(NS)]
    content = [None] * NS          # unit whose rows a stage holds
    released = [True] * NS         # the consumer of `content` has released it
    in_flight = []                 # (stage, unit) copies issued, not landed
    nxt_p = 0                      # producer's next unit
    nxt_c = list(range(G))         # each group's next unit
    weight = [rng.uniform(0.05, 1.0) for _ in range(G + 2)]
    bad = []
    while nxt_p < U or in_flight or any(u < U for u in nxt_c):
        acts = []
        if nxt_p < U:
            u, s = nxt_p, nxt_p % NS
            n = u // NS
            if n == 0 or empty[s].passes((n - 1) & 1):
                acts.append(("issue", weight[G]))
        if in_flight:
            acts.append(("land", weight[G + 1]))
        for g in range(G):
            u = nxt_c[g]
            if u < U and full[u % NS].passes((u // NS) & 1):
                acts.append((g, weight[g]))
        if not acts:
            return bad + ["deadlock"]
        act = rng.choices([a for a, _ in acts], [w for _, w in acts])[0]
        if act == "issue":
            in_flight.append((nxt_p % NS, nxt_p))
            nxt_p += 1
        elif act == "land":
            s, u = in_flight.pop(rng.randrange(len(in_flight)))
            if not released[s]:
                bad.append(f"unit {u} overwrote stage {s} (unit {content[s]}) before release")
            content[s], released[s] = u, False
            full[s].arrive()
        else:
            g, u = act, nxt_c[act]
            s = u % NS
            if content[s] != u:
                bad.append(f"group {g} read unit {content[s]} for unit {u} from stage {s}")
            released[s] = True
            empty[s].arrive()
            nxt_c[g] += G
    return bad


def run_slots(NP, NSL, nrb, G, heads, seed):
    """NP prep warps filling NSL vector slots and G consumer groups reading
    them (nrb units per head); returns the violations seen."""
    rng = random.Random(seed)
    vfull = [Barrier() for _ in range(NSL)]
    vempty = [Barrier(nrb) for _ in range(NSL)]
    content = [None] * NSL
    readers_left = [0] * NSL       # units of `content` not yet consumed
    nxt_w = list(range(NP))        # each prep warp's next head
    nxt_c = list(range(G))         # each group's next unit
    U = heads * nrb
    weight = [rng.uniform(0.05, 1.0) for _ in range(NP + G)]
    bad = []
    while any(h < heads for h in nxt_w) or any(u < U for u in nxt_c):
        acts = []
        for w in range(NP):
            li = nxt_w[w]
            if li < heads and (li < NSL or vempty[li % NSL].passes(((li // NSL) - 1) & 1)):
                acts.append((("prep", w), weight[w]))
        for g in range(G):
            u = nxt_c[g]
            if u < U:
                li = u // nrb
                if vfull[li % NSL].passes((li // NSL) & 1):
                    acts.append((("cons", g), weight[NP + g]))
        if not acts:
            return bad + ["deadlock"]
        (kind, i) = rng.choices([a for a, _ in acts], [w for _, w in acts])[0]
        if kind == "prep":
            li = nxt_w[i]
            s = li % NSL
            if readers_left[s]:
                bad.append(f"warp {i} wrote head {li} over head {content[s]} in slot {s}")
            content[s], readers_left[s] = li, nrb
            vfull[s].arrive()
            nxt_w[i] += NP
        else:
            u = nxt_c[i]
            li = u // nrb
            s = li % NSL
            if content[s] != li:
                bad.append(f"group {i} read head {content[s]} for head {li} from slot {s}")
            else:
                readers_left[s] -= 1
            vempty[s].arrive()
            nxt_c[i] += G
    return bad


def slot_rule(NP, nrb, G=4, cap=16):
    """Vector slots as the delta kernel sizes them: at least NP + 4, a
    multiple of NP, with NSL * nrb a multiple of G; 0 if none up to cap."""
    for nsl in range(NP + 4, cap + 1):
        if nsl % NP == 0 and (nsl * nrb) % G == 0:
            return nsl
    return 0


@pytest.mark.parametrize("NS", [4, 8, 12])
def test_owned_stages_hold(NS):
    for seed in range(60):
        assert run_stages(NS, 4, 90, seed) == [], (NS, seed)


def test_stages_shared_by_groups_are_caught():
    """11 stages for 4 groups: a stage's consecutive fills go to different
    groups, and some interleaving lets a group pass a parity wait on a fill
    that is not its own (the fault the ownership rule was made for)."""
    assert any(run_stages(11, 4, 90, seed) for seed in range(200))


@pytest.mark.parametrize("NP,nrb", [(8, 2), (7, 2), (6, 2), (4, 1), (6, 3), (5, 2), (1, 1)])
def test_vector_slot_rule_holds(NP, nrb):
    NSL = slot_rule(NP, nrb)
    assert NSL, (NP, nrb)
    for seed in range(60):
        assert run_slots(NP, NSL, nrb, 4, 3 * NSL + 5, seed) == [], (NP, nrb, NSL, seed)


@pytest.mark.parametrize("NP,NSL,nrb", [
    (3, 8, 1),   # NSL not a multiple of NP: one slot's fills from several warps
    (5, 12, 1),  # the same
    (4, 6, 1),   # NSL * nrb not a multiple of the groups: fills skip a group
])
def test_vector_slot_mutants_are_caught(NP, NSL, nrb):
    assert any(run_slots(NP, NSL, nrb, 4, 3 * NSL + 5, seed) for seed in range(300))


# (prep warps, depth) candidates of the tensor-core verify kernel
GRAM_CANDIDATES = [(7, 2), (6, 2), (4, 3), (4, 2), (2, 4), (6, 1), (3, 2), (2, 2), (4, 1), (2, 1)]


@pytest.mark.parametrize("NP,depth", GRAM_CANDIDATES)
def test_tensor_core_prep_stages_hold(NP, depth):
    """Every candidate at every row-block count its rule admits."""
    for nrb in (1, 2, 3):
        if (NP * depth * nrb) % 4:
            continue
        for seed in range(40):
            assert run_slots(NP, NP * depth, nrb, 4, 3 * NP * depth + 5, seed) == [], \
                (NP, depth, nrb, seed)


@pytest.mark.parametrize("NP,depth,nrb", [(7, 2, 1), (6, 1, 1), (3, 2, 1)])
def test_tensor_core_prep_stage_mutants_are_caught(NP, depth, nrb):
    """Configurations the rule excludes: some interleaving breaks them."""
    assert any(run_slots(NP, NP * depth, nrb, 4, 3 * NP * depth + 5, seed) for seed in range(300))


def run_group_rings(R, FS, G, U, seed, fold_share=0.3, flip_on_wrap=True):
    """The fused Mamba-2 step: each of G consumer groups owns a ring of R
    stages; a decode unit takes the next stage of its group's ring, a fold
    unit the next FS (the second of them, past the ring's end, waits for the
    flipped parity). The producer serves whichever group's next stage is
    free. Returns the violations seen ("deadlock" if no actor can move)."""
    rng = random.Random(seed)
    NS = G * R
    fold = [rng.random() < fold_share for _ in range(U)]
    full = [Barrier() for _ in range(NS)]
    empty = [Barrier() for _ in range(NS)]
    content = [None] * NS
    released = [True] * NS
    in_flight = []
    # producer, per group: next unit, stages of it issued, ring position,
    # parity of that position's fill, whether the ring has wrapped
    p_nxt, p_f, p_t, p_ph, p_reuse = list(range(G)), [0] * G, [0] * G, [0] * G, [False] * G
    # consumers, per group: next unit, ring position, parity
    c_nxt, c_t, c_ph = list(range(G)), [0] * G, [0] * G
    weight = [rng.uniform(0.05, 1.0) for _ in range(2 * G + 1)]
    bad = []
    while any(i < U for i in p_nxt) or in_flight or any(i < U for i in c_nxt):
        acts = []
        for g in range(G):
            if p_nxt[g] < U:
                s = g * R + p_t[g]
                if not p_reuse[g] or empty[s].passes(p_ph[g] ^ 1):
                    acts.append((("issue", g), weight[g]))
            i = c_nxt[g]
            if i < U:
                s0, ph0 = g * R + c_t[g], c_ph[g]
                wrap = c_t[g] + 1 == R
                s1 = g * R + (0 if wrap else c_t[g] + 1)
                ph1 = c_ph[g] ^ 1 if (wrap and flip_on_wrap) else c_ph[g]
                two = fold[i] and FS > 1
                if full[s0].passes(ph0) and (not two or full[s1].passes(ph1)):
                    acts.append((("consume", g), weight[G + g]))
        if in_flight:
            acts.append((("land", 0), weight[2 * G]))
        if not acts:
            return bad + ["deadlock"]
        kind, g = rng.choices([a for a, _ in acts], [w for _, w in acts])[0]
        if kind == "issue":
            i, s = p_nxt[g], g * R + p_t[g]
            in_flight.append((s, (i, p_f[g])))
            p_t[g] += 1
            if p_t[g] == R:
                p_t[g], p_ph[g], p_reuse[g] = 0, p_ph[g] ^ 1, True
            p_f[g] += 1
            if p_f[g] == (FS if fold[i] else 1):
                p_f[g] = 0
                p_nxt[g] += G
        elif kind == "land":
            s, what = in_flight.pop(rng.randrange(len(in_flight)))
            if not released[s]:
                bad.append(f"{what} overwrote stage {s} ({content[s]}) before release")
            content[s], released[s] = what, False
            full[s].arrive()
        else:
            i = c_nxt[g]
            stages = []
            for f in range(FS if fold[i] else 1):
                stages.append(g * R + c_t[g])
                c_t[g] += 1
                if c_t[g] == R:
                    c_t[g], c_ph[g] = 0, c_ph[g] ^ 1
            for f, s in enumerate(stages):
                if content[s] != (i, f):
                    bad.append(f"group {g} read {content[s]} for {(i, f)} from stage {s}")
            for s in stages:
                released[s] = True
                empty[s].arrive()
            c_nxt[g] += G
    return bad


@pytest.mark.parametrize("R,FS", [(1, 1), (2, 1), (3, 1), (2, 2), (3, 2), (5, 2)])
def test_fused_step_group_rings_hold(R, FS):
    """Rings of at least FS stages per group (the launch requires
    NS >= 4 * FS), decode and fold units mixed at random."""
    for seed in range(60):
        assert run_group_rings(R, FS, 4, 80, seed) == [], (R, FS, seed)


def test_fused_step_ring_shorter_than_a_fold_unit_is_caught():
    """One stage per group with two-stage fold units: the group would need
    both fills of its single stage at once."""
    assert any(run_group_rings(1, 2, 4, 80, seed) for seed in range(50))


def test_fused_step_second_stage_parity_is_needed():
    """A fold unit whose second stage lies past the ring's end must wait for
    the flipped parity; waiting for the first stage's parity passes on the
    previous fill of that stage."""
    assert any(run_group_rings(3, 2, 4, 80, seed, flip_on_wrap=False) for seed in range(200))
