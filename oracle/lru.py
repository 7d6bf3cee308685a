"""Per-step LRU slot table of the GPU expert cache (oracle; test
infrastructure only).

Pages.  FreeToken keeps experts in a global LRU expert cache in GPU memory;
most routed experts of a decode step hit it and the misses are loaded into it
("FreeToken：把 284B MoE 塞进游戏 PC", zhichai.net, §二, the "Decode" and "LRU
为什么赢" paragraphs; juejin.cn overview §二, 全局 LRU 专家缓存).  The pages do
not say how one step's accesses are ordered.  Reading taken:

* U = the distinct experts routed in the step.  They are accessed hits first
  (experts already resident, ascending id), then misses (ascending id).
* A hit becomes most recently used.  A miss takes the lowest-index free slot
  if there is one, otherwise it evicts the least recently used expert; then
  it becomes most recently used.
* Hits first means no expert needed in a step is evicted by that step while
  |U| <= slots.  When |U| > slots the same rule evicts the step's own earliest
  accesses; any two accesses that share a slot are then at least ``slots``
  apart in the access order.

This is the textbook slot table: each slot keeps a recency stamp from a
counter that ticks once per access; the LRU victim is the occupied slot with
the smallest stamp.
"""
from __future__ import annotations

from typing import List, Sequence, Tuple


class SlotTable:
    def __init__(self, E: int, S: int):
        self.E, self.S = E, S
        self.slot_of = [-1] * E
        self.expert_of = [-1] * S
        self.stamp = [0] * S
        self.clock = 0

    def install(self, e: int, s: int) -> None:
        """Put expert e into slot s as most recently used (a load of the
        cache outside a step, e.g. a prefill layer that holds every expert)."""
        if self.slot_of[e] >= 0:
            self.expert_of[self.slot_of[e]] = -1
        old = self.expert_of[s]
        if old >= 0:
            self.slot_of[old] = -1
        self.expert_of[s] = e
        self.slot_of[e] = s
        self.clock += 1
        self.stamp[s] = self.clock

    def step(self, routed: Sequence[int]) -> List[Tuple[int, int, bool, int]]:
        """Apply one step.  Returns the access list [(expert, slot, hit,
        evicted expert or -1)] in access order."""
        U = sorted(set(int(e) for e in routed))
        hits = [e for e in U if self.slot_of[e] >= 0]
        misses = [e for e in U if self.slot_of[e] < 0]
        out = []
        for e in hits:
            s = self.slot_of[e]
            self.clock += 1
            self.stamp[s] = self.clock
            out.append((e, s, True, -1))
        for e in misses:
            free = [s for s in range(self.S) if self.expert_of[s] < 0]
            if free:
                s = free[0]
            else:
                s = min(range(self.S), key=lambda q: self.stamp[q])
            ev = self.expert_of[s]
            if ev >= 0:
                self.slot_of[ev] = -1
            self.expert_of[s] = e
            self.slot_of[e] = s
            self.clock += 1
            self.stamp[s] = self.clock
            out.append((e, s, False, ev))
        return out

    def resize(self, S_new: int) -> None:
        """Change the number of slots between steps without reloading any
        expert (the pages' elastic expert cache, zhichai.net, §二 "弹性显存":
        the GPU expert cache is resized at scheduler safe points).  Reading
        taken: the min(S_new, occupied) most recently used experts stay, with
        their recency stamps; they move to slots 0, 1, ... in the order of
        their old slots; the other slots are free; the clock is unchanged."""
        occ = [s for s in range(self.S) if self.expert_of[s] >= 0]
        keep = sorted(sorted(occ, key=lambda s: self.stamp[s], reverse=True)[:S_new])
        experts = [self.expert_of[s] for s in keep]
        stamps = [self.stamp[s] for s in keep]
        self.S = S_new
        self.slot_of = [-1] * self.E
        self.expert_of = [-1] * S_new
        self.stamp = [0] * S_new
        for i, (e, st) in enumerate(zip(experts, stamps)):
            self.expert_of[i] = e
            self.stamp[i] = st
            self.slot_of[e] = i

    def recency(self) -> List[int]:
        """Occupied slots from least to most recently used."""
        occ = [s for s in range(self.S) if self.expert_of[s] >= 0]
        return sorted(occ, key=lambda s: self.stamp[s])
