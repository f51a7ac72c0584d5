"""Plain CPU oracle of owner placement (test infrastructure only).

TEST INFRASTRUCTURE ONLY: imported by ``tests/`` alone; the library never
imports, links or calls it and shares no code with it.

DMuon technical summary (gist.science 2606.27153), §2.3 "compute-aware load
balancing": every 2-D matrix gets exactly one owner rank.  The assignment
minimises the predicted makespan, which is the largest total cost on any owner.
The pages solve this exactly (a MILP) where the search is small. Otherwise they
use a greedy heuristic.

Readings where the pages are silent:

* The greedy is longest-processing-time first (LPT). Take the matrices in
  decreasing cost, and give each to the owner whose total is smallest so far.
  Equal costs go in input order; equal totals go to the lower rank.
* The exact answer is the minimum makespan over all world**count assignments.
  Several assignments can reach it, so only the makespan is unique.
"""
from __future__ import annotations

import itertools


def makespan(cost, owner, world):
    """Largest total cost over the `world` owners."""
    load = [0.0] * world
    for c, r in zip(cost, owner):
        load[r] += c
    return max(load) if world else 0.0


def lpt(cost, world):
    """Greedy longest-processing-time assignment: list of owner ranks."""
    order = sorted(range(len(cost)), key=lambda i: (-cost[i], i))
    load = [0.0] * world
    owner = [0] * len(cost)
    for i in order:
        r = min(range(world), key=lambda q: (load[q], q))
        owner[i] = r
        load[r] += cost[i]
    return owner


def optimal_makespan(cost, world):
    """Minimum makespan by enumerating every assignment (tiny inputs only)."""
    best = float("inf")
    for owner in itertools.product(range(world), repeat=len(cost)):
        best = min(best, makespan(cost, owner, world))
    return best if cost else 0.0
