"""Pins of the oracle's expert-slot pool simulator (no GPU)."""
import json
import os

import numpy as np
import pytest

import oracle

GOLD = os.path.join(os.path.dirname(__file__), "golden", "lru_trace.json")


def test_hand_worked_trace():
    g = json.load(open(GOLD))
    misses, table = oracle.pool_sim(g["E"], g["S"], g["steps"])
    assert misses.tolist() == g["misses"]
    assert table.tolist() == g["final_table"]


def test_step_larger_than_pool_is_rejected():
    with pytest.raises(ValueError):
        oracle.pool_sim(6, 3, [[0, 1, 2, 3]])


def test_full_pool_never_misses():
    rng = np.random.default_rng(0)
    steps = [rng.choice(32, size=5, replace=False).tolist() for _ in range(50)]
    misses, table = oracle.pool_sim(32, 32, steps, init_full=True)
    assert len(misses) == 0 and table.tolist() == list(range(32))


@pytest.mark.parametrize("seed", range(5))
def test_invariants_on_random_traces(seed):
    """Misses only for non-resident experts, never evicting a slot the step
    uses, at most S resident, and a cold pool misses exactly once per
    distinct expert while it still has room."""
    rng = np.random.default_rng(seed)
    E, S = 40, 12
    p = 1.0 / np.arange(1, E + 1) ** 1.1
    p /= p.sum()
    steps = [sorted(set(rng.choice(E, size=4, p=p).tolist())) for _ in range(200)]
    misses, table = oracle.pool_sim(E, S, steps)
    resident = {}
    owner = {}
    it = 0
    seen = set()
    for n, sel in enumerate(steps, start=1):
        step_m = []
        while it < len(misses) and misses[it][0] == n:
            step_m.append(misses[it].tolist())
            it += 1
        missed = [e for _, e, _ in step_m]
        assert missed == sorted(e for e in sel if e not in resident)
        for _, e, s in step_m:
            assert owner.get(s) not in sel  # never evict a slot this step needs
            if s in owner:
                del resident[owner[s]]
            owner[s] = e
            resident[e] = s
        assert len(resident) <= S
        if len(seen | set(sel)) <= S:
            assert len(step_m) == len(set(sel) - seen)
        seen |= set(sel)
    assert it == len(misses)
    assert all(table[e] == resident.get(e, -1) for e in range(E))


def test_hand_worked_seeded_trace():
    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "lru_seeded_trace.json")))
    misses, table = oracle.pool_sim(g["E"], g["S"], g["steps"], seed=g["seed"])
    assert misses.tolist() == g["misses"]
    assert table.tolist() == g["final_table"]


def test_seeding_the_experts_a_step_needs_removes_its_misses():
    rng = np.random.default_rng(3)
    E, S = 40, 12
    steps = [sorted(rng.choice(E, size=6, replace=False).tolist()) for _ in range(30)]
    cold, _ = oracle.pool_sim(E, S, steps)
    warm, _ = oracle.pool_sim(E, S, steps, seed=steps[0])
    assert not any(m[0] == 1 for m in warm)  # the first step only hits
    assert len(warm) <= len(cold)
    # seeding every expert of a full-size pool is init_full with another order
    none, _ = oracle.pool_sim(E, E, steps, seed=list(range(E))[::-1])
    assert len(none) == 0


def test_invalid_seeds_are_rejected():
    for seed in ([0, 0], [7], [0, 1, 2, 3]):
        with pytest.raises(ValueError):
            oracle.pool_sim(6, 3, [[0]], seed=seed)
