"""Placement-policy replay (host logic, no GPU): pinned against the oracle's
LRU and the closed forms of the static placements."""
import random

from oracle.lru import SlotTable
from routed_expert_layer_gemv_gb300 import placement as pl


def _trace(rng, E, k, steps, batch):
    return [[rng.randrange(E) for _ in range(batch * k)] for _ in range(steps)]


def test_lru_replay_matches_the_oracle_slot_table():
    rng = random.Random(3)
    for _ in range(60):
        E = rng.randint(2, 80)
        S = rng.randint(1, E)
        k = rng.randint(1, min(8, E))
        cache, T = pl.LRUCache(E, S), SlotTable(E, S)
        for step in _trace(rng, E, k, 40, rng.randint(1, 8)):
            m = cache.step(step)
            acc = T.step(step)
            assert m == sum(1 for a in acc if not a[2])
            assert cache.expert_of == T.expert_of and cache.stamp == T.stamp and cache.clock == T.clock


def test_everything_fits():
    # n_slots >= E: LRU misses each expert once (its first use), static placements never
    rng = random.Random(5)
    E = 12
    trace = _trace(rng, E, 3, 30, 2)
    res = pl.replay(trace, E, E, trace[:4])
    assert res["lru"]["misses"] == len(set(e for s in trace for e in s))
    assert res["prefill_static"]["misses"] == 0 and res["blind_static"]["misses"] == 0


def test_static_placements_by_brute_force():
    rng = random.Random(9)
    E, S = 30, 7
    trace = _trace(rng, E, 4, 50, 3)
    prefill = _trace(rng, E, 4, 20, 1)
    res = pl.replay(trace, E, S, prefill)
    count = {e: sum(r.count(e) for r in prefill) for e in range(E)}
    top = sorted(sorted(range(E), key=lambda e: (-count[e], e))[:S])
    assert pl.prefill_static_set(prefill, E, S) == top
    n_distinct = sum(len(set(s)) for s in trace)
    for name, resident in (("prefill_static", set(top)), ("blind_static", set(range(S)))):
        want = sum(len(set(s) - resident) for s in trace)
        assert res[name]["misses"] == want and res[name]["distinct"] == n_distinct
        assert abs(res[name]["miss_rate"] - want / n_distinct) < 1e-15


def test_prefill_ranking_ties_to_lower_id():
    # experts 4 and 2 are routed twice, 7 and 1 once: top-3 = {2, 4} + the lower of {1, 7}
    assert pl.prefill_static_set([[4, 2], [4, 7], [2, 1]], 8, 3) == [1, 2, 4]
