"""The balanced schedule's arithmetic, restated in Python and checked for the
invariants the partial merges rely on (host-side specification test).

The tile kernel's producer numbers every (sequence, KV head) unit's visible
chunks globally, with `seg_cost` virtual chunks ahead of each unit's real
ones, and CTA c takes positions [c*N/C, (c+1)*N/C). A unit whose real chunks
span CTAs c1..c2 is split; CTA c writes its partial into slot 2c for the unit
it starts with and 2c + 1 for the one it ends with, and the merge reads the
slots s0, sbase + k*sstride (k >= 1). This file restates that arithmetic
(the device code is pa_tile.cuh: sched_start, sched_owner, balanced_desc and
Producer::run) and checks, over random length mixes, CTA counts and segment
costs, that

  * every real chunk of every unit is streamed by exactly one CTA,
  * a unit covered by one CTA is written directly (no slot),
  * no two partials share a slot,
  * each split unit's slots are exactly the merge descriptor's list, in
    partition order,
  * a CTA holds at most two split segments.
"""

import random

import pytest


def start(c, N, C):
    return c * N // C


def owner(x, N, C):
    return ((x + 1) * C - 1) // N


def schedule(chunks_per_unit, C0, A):
    """Segments (unit, first chunk, end chunk, slot or None) per CTA, and the
    merge descriptor (nseg, s0, sbase, sstride) per unit."""
    nb = [max(1, n) for n in chunks_per_unit]
    w = [n + A for n in nb]
    P = [0] * len(nb)
    for u in range(1, len(nb)):
        P[u] = P[u - 1] + w[u - 1]
    N = sum(w)
    C = min(C0, N)

    def desc(u):
        c1, c2 = owner(P[u] + A, N, C), owner(P[u] + A + nb[u] - 1, N, C)
        return (c2 - c1 + 1, 2 * c1 + (1 if start(c1, N, C) < P[u] else 0), 2 * c1, 2)

    segs = {}
    for c in range(C):
        x, x1 = start(c, N, C), start(c + 1, N, C)
        out = []
        u = next(i for i in range(len(nb)) if P[i] <= x < P[i] + w[i]) if x < x1 else len(nb)
        while x < x1:
            R0 = P[u] + A
            lo, hi = max(x, R0), min(x1, R0 + nb[u])
            if lo < hi:
                d = desc(u)
                slot = None
                if d[0] > 1:
                    slot = 2 * c + (1 if (c == owner(R0, N, C) and start(c, N, C) < P[u]) else 0)
                out.append((u, lo - R0, hi - R0, slot))
            x = P[u] + w[u]
            u += 1
        segs[c] = out
    return segs, {u: desc(u) for u in range(len(nb))}, nb


def check(chunks_per_unit, C0, A):
    segs, descs, nb = schedule(chunks_per_unit, C0, A)
    cover = [[0] * n for n in nb]
    slots_of = {u: [] for u in range(len(nb))}
    used = set()
    for c, out in segs.items():
        assert sum(1 for s in out if s[3] is not None) <= 2
        for u, k0, k1, slot in out:
            for k in range(k0, k1):
                cover[u][k] += 1
            if slot is not None:
                assert slot not in used, f"slot {slot} written twice"
                used.add(slot)
                slots_of[u].append(slot)
    for u, d in descs.items():
        assert all(v == 1 for v in cover[u]), f"unit {u} coverage {cover[u]}"
        nseg, s0, sbase, sstride = d
        if nseg == 1:
            assert slots_of[u] == []
        else:
            expect = [s0] + [sbase + k * sstride for k in range(1, nseg)]
            assert slots_of[u] == expect, (u, slots_of[u], expect)


@pytest.mark.parametrize("seg_cost", [0, 1, 2, 4])
def test_balanced_schedule_invariants(seg_cost):
    rng = random.Random(1234 + seg_cost)
    for _ in range(1500):
        units = [rng.choice([0, 0, 1, 2, 3, rng.randint(1, 90)]) for _ in range(rng.randint(1, 40))]
        C0 = rng.choice([1, 2, 3, 5, 7, 16, 64, 152, 304, 1000])
        check(units, C0, seg_cost)


def test_segment_cost_moves_chunks_off_many_unit_ctas():
    """With a segment cost, a CTA whose range holds many short units streams
    fewer real chunks than one inside a long unit."""
    units = [2] * 40 + [400]
    segs, _, _ = schedule(units, 8, 1)
    real = {c: sum(k1 - k0 for _, k0, k1, _ in out) for c, out in segs.items()}
    first, last = real[0], real[7]
    assert len(segs[0]) > 5 and len(segs[7]) == 1
    assert first < last
