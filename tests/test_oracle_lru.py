"""Pin of the oracle's stamp-based LRU slot table against a naive list
simulation (no GPU)."""
import numpy as np
import pytest

from conftest import ORACLES, swap_oracle

from oracle.lru import SlotTable


@pytest.fixture(autouse=True, params=ORACLES)
def oracle_impl(request, monkeypatch):
    return swap_oracle(__name__, request, monkeypatch, ("SlotTable",))



class NaiveLRU:
    """Recency kept as a Python list of experts, least recent first."""

    def __init__(self, E, S):
        self.S = S
        self.where = {}          # expert -> slot
        self.order = []          # experts, LRU first

    def step(self, routed):
        U = sorted(set(routed))
        hits = [e for e in U if e in self.where]
        misses = [e for e in U if e not in self.where]
        acc = []
        for e in hits:
            self.order.remove(e)
            self.order.append(e)
            acc.append((e, self.where[e], True, -1))
        for e in misses:
            used = set(self.where.values())
            free = [s for s in range(self.S) if s not in used]
            ev = -1
            if free:
                s = free[0]
            else:
                ev = self.order.pop(0)
                s = self.where.pop(ev)
            self.where[e] = s
            self.order.append(e)
            acc.append((e, s, False, ev))
        return acc

    def expert_of(self):
        out = [-1] * self.S
        for e, s in self.where.items():
            out[s] = e
        return out


@pytest.mark.parametrize("E,S,per_step", [(8, 3, 2), (128, 47, 8), (128, 47, 40), (256, 28, 20), (16, 16, 5)])
def test_slot_table_matches_naive_list(E, S, per_step):
    g = np.random.default_rng(E * 1000 + S)
    T, N = SlotTable(E, S), NaiveLRU(E, S)
    hot = g.choice(E, min(E, 2 * S), replace=False)
    for step in range(300):
        pool = hot if g.random() < 0.7 else np.arange(E)
        routed = g.choice(pool, min(per_step, len(pool)), replace=False)
        a1, a2 = T.step(routed), N.step(list(routed))
        assert a1 == a2
        assert T.expert_of == N.expert_of()
        assert [T.expert_of[s] for s in T.recency()] == N.order


def test_shared_slot_accesses_are_at_least_S_apart():
    g = np.random.default_rng(1)
    E, S = 128, 47
    T = SlotTable(E, S)
    for _ in range(50):
        acc = T.step(g.choice(E, 100, replace=False))
        last = {}
        for i, (_, s, _, _) in enumerate(acc):
            if s in last:
                assert i - last[s] >= S
            last[s] = i


def test_install_then_hit():
    T = SlotTable(4, 2)
    T.install(3, 1)
    T.install(0, 0)
    acc = T.step([3, 2])
    assert acc == [(3, 1, True, -1), (2, 0, False, 0)]
    assert T.recency() == [1, 0]


class NaiveLRUResizable(NaiveLRU):
    def resize(self, S):
        # keep the S most recently used (the end of the order list), then
        # give them slots 0, 1, ... in the order of their old slots
        kept = self.order[-S:] if S > 0 else []
        by_slot = sorted(kept, key=lambda e: self.where[e])
        self.S = S
        self.where = {e: i for i, e in enumerate(by_slot)}
        self.order = [e for e in self.order if e in self.where]


@pytest.mark.parametrize("E,S,per_step", [(16, 6, 3), (128, 47, 8), (256, 28, 20)])
def test_resize_matches_naive_list(E, S, per_step):
    g = np.random.default_rng(E + 7 * S)
    T, N = SlotTable(E, S), NaiveLRUResizable(E, S)
    cur = S
    for step in range(200):
        if step % 23 == 22:
            cur = int(g.integers(1, E + 1))
            T.resize(cur)
            N.resize(cur)
            assert T.expert_of == N.expert_of()
            assert [T.expert_of[s] for s in T.recency()] == N.order
        routed = g.choice(E, min(per_step, E), replace=False)
        assert T.step(routed) == N.step(list(routed))
        assert T.expert_of == N.expert_of()
        assert [T.expert_of[s] for s in T.recency()] == N.order


def test_resize_keeps_stamps_and_clock():
    T = SlotTable(8, 4)
    for routed in ([0, 1], [2, 3], [4], [1]):
        T.step(routed)
    clk, stamps = T.clock, dict(zip(T.expert_of, T.stamp))
    # 4 evicted 0 from slot 0, so the two most recent are 4 (slot 0, stamp 5)
    # and 1 (slot 1, stamp 6), kept in that slot order
    T.resize(2)
    assert T.expert_of == [4, 1] and T.clock == clk
    assert T.stamp == [stamps[4], stamps[1]]
    T.resize(5)                       # growing: same experts, new free slots
    assert T.expert_of == [4, 1, -1, -1, -1] and T.clock == clk
