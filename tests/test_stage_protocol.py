"""A host model of the quantizer's stage ring when a column-only launch splits
each CTA's tiles between two warp groups (even tiles, odd tiles).

Each stage has one mbarrier; a load that lands completes one phase, and a
wait on parity q passes once the completed-phase count has parity != q (the
hardware's parity test).  A group waits for tile t on stage t % NSTG with
parity (t // NSTG) & 1, reads it, and releases it; the release of a tile
issues the load of tile t + NSTG into the same stage.  The model checks that
a group never passes a wait before the load of its own tile has landed.
With an odd stage count the two groups share stages and a group can pass on
the other group's phase; with an even count each stage serves one group.
"""

import random

import pytest


def run_schedule(nstg: int, ntiles: int, seed: int) -> bool:
    """One random interleaving of loads landing and groups progressing.
    Returns False if a group passed a wait on a stage that did not hold its
    tile's completed load."""
    rnd = random.Random(seed)
    completed = [0] * nstg            # completed phases per stage
    inflight = {}                     # stage -> tile whose load is in flight
    landed = [None] * nstg            # tile whose load last landed in each stage
    for t in range(min(nstg, ntiles)):
        inflight[t % nstg] = t
    nxt = [0, 1]                      # next tile of each group
    while nxt[0] < ntiles or nxt[1] < ntiles:
        if inflight and rnd.random() < 0.4:
            s = rnd.choice(sorted(inflight))
            landed[s] = inflight.pop(s)
            completed[s] += 1
            continue
        g = rnd.randrange(2)
        t = nxt[g]
        if t >= ntiles:
            continue
        s, use = t % nstg, t // nstg
        if (completed[s] & 1) == (use & 1):          # the parity wait does not pass yet
            continue
        if landed[s] != t or s in inflight:
            return False                              # passed on another tile's phase
        if t + nstg < ntiles:
            inflight[s] = t + nstg                    # release: the stage's next load
        nxt[g] += 2
    return True


@pytest.mark.parametrize("nstg", [2, 4])
def test_even_stage_counts_never_alias(nstg):
    assert all(run_schedule(nstg, 40, seed) for seed in range(2000))


def test_three_stages_alias():
    """The configuration the kernel's compile-time check rules out."""
    assert sum(not run_schedule(3, 40, seed) for seed in range(2000)) > 1000
