"""Owner placement: the oracle's pins, then the library against the oracle.

Host-only code, so everything here runs on CPU.  The oracle (plain Python
LPT and brute-force optimum) is pinned by Graham's worst-case instance and
bound, and by special cases with known answers.  The library's LPT must
match the oracle's assignment exactly; its exact solver must reach the
brute-force optimal makespan (the only unique part of an optimal assignment).
"""
import math
import random

import pytest

from oracle import partition as P

# ---------------------------------------------------------------- oracle pins


def graham_instance(w):
    """Graham (1969): 2w+1 jobs 2w-1, 2w-1, 2w-2, 2w-2, ..., w+1, w+1, w, w, w.
    LPT's makespan is 4w-1 and the optimum is 3w, so LPT meets its bound
    4/3 - 1/(3w) with equality."""
    cost = []
    for v in range(2 * w - 1, w, -1):
        cost += [v, v]
    return cost + [w, w, w]


@pytest.mark.parametrize("w", [2, 3])
def test_oracle_graham_worst_case(w):
    cost = graham_instance(w)
    assert P.makespan(cost, P.lpt(cost, w), w) == 4 * w - 1
    assert P.optimal_makespan(cost, w) == 3 * w
    assert (4 * w - 1) / (3 * w) == pytest.approx(4 / 3 - 1 / (3 * w))


def test_oracle_lpt_within_graham_bound_on_random_instances():
    rng = random.Random(5)
    for _ in range(150):
        w = rng.randint(2, 3)
        n = rng.randint(1, 7)
        cost = [rng.choice([rng.randint(1, 20), rng.random() * 10]) for _ in range(n)]
        opt = P.optimal_makespan(cost, w)
        got = P.makespan(cost, P.lpt(cost, w), w)
        assert opt - 1e-12 <= got <= (4 / 3 - 1 / (3 * w)) * opt + 1e-9
        assert opt >= max(max(cost), sum(cost) / w) - 1e-12


def test_oracle_special_cases():
    # equal costs: round robin in input order
    assert P.lpt([1.0] * 7, 3) == [0, 1, 2, 0, 1, 2, 0]
    # one owner takes everything
    assert P.lpt([3.0, 1.0, 2.0], 1) == [0, 0, 0]
    # no more matrices than owners: one each, heaviest to rank 0
    assert P.lpt([1.0, 5.0, 3.0], 4) == [2, 0, 1]
    assert P.optimal_makespan([1.0, 5.0, 3.0], 4) == 5.0
    # worked by hand: 7,5,4,3,1 on two owners -> LPT {7,3}{5,4,1}: 10; optimum 10
    assert P.lpt([7, 5, 4, 3, 1], 2) == [0, 1, 1, 0, 1]
    assert P.optimal_makespan([7, 5, 4, 3, 1], 2) == 10
    assert P.lpt([], 3) == [] and P.optimal_makespan([], 3) == 0.0


def _spt(cost, world):  # planted slip: lightest first
    order = sorted(range(len(cost)), key=lambda i: (cost[i], i))
    load = [0.0] * world
    owner = [0] * len(cost)
    for i in order:
        r = min(range(world), key=lambda q: (load[q], q))
        owner[i] = r
        load[r] += cost[i]
    return owner


def _most_loaded(cost, world):  # planted slip: most-loaded owner
    order = sorted(range(len(cost)), key=lambda i: (-cost[i], i))
    load = [0.0] * world
    owner = [0] * len(cost)
    for i in order:
        r = max(range(world), key=lambda q: (load[q], -q))
        owner[i] = r
        load[r] += cost[i]
    return owner


@pytest.mark.parametrize("slip", [_spt, _most_loaded])
def test_planted_slips_break_a_pin(slip):
    """Each plausible mistake in the greedy fails the Graham bound somewhere."""
    rng = random.Random(11)
    broken = False
    for _ in range(300):
        w = rng.randint(2, 3)
        cost = [rng.randint(1, 30) for _ in range(rng.randint(3, 7))]
        opt = P.optimal_makespan(cost, w)
        if P.makespan(cost, slip(cost, w), w) > (4 / 3 - 1 / (3 * w)) * opt + 1e-9:
            broken = True
            break
    assert broken


# ---------------------------------------------------------------- library

def _lib():
    import newton_schulz_04_gb300 as m
    from newton_schulz_04_gb300 import build as b
    b.build()
    return m


def test_library_lpt_matches_oracle_exactly():
    m = _lib()
    rng = random.Random(7)
    for _ in range(300):
        w = rng.randint(1, 9)
        n = rng.randint(0, 60)
        # small integer costs force many ties in both sort order and loads
        cost = [float(rng.randint(0, 6)) if rng.random() < 0.6 else rng.random() * 4 for _ in range(n)]
        owner, load = m.partition(cost, w, exact_limit=0)
        assert owner == P.lpt(cost, w)
        ref = [0.0] * w
        for c, r in zip(cost, owner):
            ref[r] += c
        assert load == pytest.approx(ref, abs=0, rel=1e-15)


def test_library_exact_solver_reaches_the_optimum():
    m = _lib()
    rng = random.Random(8)
    for _ in range(120):
        w = rng.randint(2, 3)
        n = rng.randint(1, 8)
        cost = [float(rng.randint(1, 25)) if rng.random() < 0.5 else rng.random() * 10 for _ in range(n)]
        owner, load = m.partition(cost, w, exact_limit=24)
        assert all(0 <= r < w for r in owner) and len(owner) == n
        assert max(load) == pytest.approx(P.optimal_makespan(cost, w), rel=1e-12)
        assert max(load) <= P.makespan(cost, P.lpt(cost, w), w) + 1e-12
    for w in (2, 3):  # LPT's worst case: the exact solver recovers 3w
        owner, load = m.partition([float(c) for c in graham_instance(w)], w, exact_limit=24)
        assert max(load) == 3 * w


def test_library_partition_is_deterministic_and_scales():
    m = _lib()
    rng = random.Random(9)
    cost = [rng.random() for _ in range(5000)]
    a = m.partition(cost, 8, exact_limit=12)
    b = m.partition(list(cost), 8, exact_limit=12)
    assert a == b
    owner, load = a
    # list-scheduling bound: makespan <= total / w + max cost
    assert max(load) <= sum(cost) / 8 + max(cost) + 1e-9
    assert sorted(set(owner)) == list(range(8))


def test_library_partition_rejects_bad_arguments():
    m = _lib()
    with pytest.raises(m.MuonError):
        m.partition([1.0, -1.0], 2)
    with pytest.raises(m.MuonError):
        m.partition([1.0, math.nan], 2)
    with pytest.raises(m.MuonError):
        m.partition([1.0, math.inf], 2)
    with pytest.raises(m.MuonError):
        m.partition([1.0], 0)
    with pytest.raises(m.MuonError):
        m.partition([1.0], 2, exact_limit=25)
    assert m.partition([], 3) == ([], [0.0, 0.0, 0.0])


def test_cost_estimate_properties():
    m = _lib()
    c = m.cost_estimate([(4096, 4096), (4096, 14336), (14336, 4096), (1024, 1024), (256, 1024)])
    assert all(x > 0 for x in c)
    assert c[1] == c[2]                      # orientation does not change the work
    assert c[0] < c[1]                       # a longer long side costs more
    assert c[3] < c[0] and c[4] < c[3]
    # square: five steps of SYRK + A A + B X on 4096^2 execute ~2e12 flops
    assert 0.3e-3 < c[0] < 3e-3
    more = m.cost_estimate([(4096, 4096)], steps=10)
    assert more[0] > 1.5 * c[0]            # twice the steps, well over 1.5 times the work
    torch = __import__("torch")
    f32 = m.cost_estimate([(4096, 4096)], dtype=torch.float32)
    assert 2.5 * c[0] < f32[0] < 4 * c[0]    # fp16 pairs: three products per product
    f32_long = m.cost_estimate([(4096, 4096)], steps=10, dtype=torch.float32)
    assert f32_long[0] > 10 * more[0]        # beyond 6 steps fp32 runs on FFMA
    zero = m.cost_estimate([(4096, 4096)], steps=0)
    assert zero[0] < c[0] / 12               # pack + apply only (~370 MB of traffic)
    with pytest.raises(m.MuonError):
        m.cost_estimate([(0, 16)])
    assert m.cost_estimate([]) == []


def test_owned_covers_every_matrix_once():
    m = _lib()
    shapes = [(4096, 4096)] * 4 + [(4096, 14336)] * 2 + [(14336, 4096)] + [(1024, 3072)] * 5
    for world in (1, 2, 3, 8):
        got = sorted(i for r in range(world) for i in m.owned(shapes, r, world))
        assert got == list(range(len(shapes)))
