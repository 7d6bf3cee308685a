"""The per-step LRU slot table of the expert cache, by the C++ oracle, with
the numpy oracle's names (see oracle/lru.py for the reading).  Test
infrastructure only."""
from __future__ import annotations

import ctypes as C
from typing import List, Sequence, Tuple

import numpy as np

from . import arr, lib, ptr


class SlotTable:
    def __init__(self, E: int, S: int):
        self.E, self.S = E, S
        self._h = lib().orc_lru_new(E, S)

    def __del__(self):
        try:
            if self._h:
                lib().orc_lru_free(self._h)
                self._h = None
        except Exception:
            pass

    def _state(self):
        eo = np.empty(self.S, dtype=np.int32)
        st = np.empty(self.S, dtype=np.uint64)
        so = np.empty(self.E, dtype=np.int32)
        clk = C.c_ulonglong(0)
        lib().orc_lru_state(self._h, ptr(eo, C.c_int), ptr(st, C.c_ulonglong), C.byref(clk), ptr(so, C.c_int))
        return eo, st, int(clk.value), so

    @property
    def expert_of(self) -> List[int]:
        return [int(v) for v in self._state()[0]]

    @property
    def stamp(self) -> List[int]:
        return [int(v) for v in self._state()[1]]

    @property
    def clock(self) -> int:
        return self._state()[2]

    @property
    def slot_of(self) -> List[int]:
        return [int(v) for v in self._state()[3]]

    def install(self, e: int, s: int) -> None:
        lib().orc_lru_install(self._h, int(e), int(s))

    def step(self, routed: Sequence[int]) -> List[Tuple[int, int, bool, int]]:
        r = arr(np.asarray(routed).reshape(-1), np.int32)
        n = r.size
        ae, as_, ah, av = (np.empty(max(n, 1), dtype=np.int32) for _ in range(4))
        U = lib().orc_lru_step(self._h, ptr(r, C.c_int), n, ptr(ae, C.c_int), ptr(as_, C.c_int), ptr(ah, C.c_int),
                               ptr(av, C.c_int))
        return [(int(ae[i]), int(as_[i]), bool(ah[i]), int(av[i])) for i in range(U)]

    def drop(self, e: int) -> None:
        """Take expert e out of the table (its slot becomes free; stamps and
        clock unchanged) -- the cache after a fill of e that failed."""
        eo, st, clk, so = self._state()
        if so[e] >= 0:
            eo[so[e]] = -1
            lib().orc_lru_set(self._h, ptr(arr(eo, np.int32), C.c_int), ptr(arr(st, np.uint64), C.c_ulonglong), clk)

    def resize(self, S_new: int) -> None:
        """Between steps: the min(S_new, occupied) most recently used experts
        stay (stamps kept), in slots 0, 1, ... by old slot order."""
        lib().orc_lru_resize(self._h, int(S_new))
        self.S = int(S_new)

    def recency(self) -> List[int]:
        """Occupied slots from least to most recently used."""
        eo, st, _, _ = self._state()
        occ = [s for s in range(self.S) if eo[s] >= 0]
        return sorted(occ, key=lambda s: int(st[s]))
