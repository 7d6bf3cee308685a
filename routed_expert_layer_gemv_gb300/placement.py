"""Expert placement policies replayed over decode routing traces (host only).

The layer's expert cache is a global LRU over n_slots slots.  One step of it
takes the step's distinct routed experts, hits in ascending id and then misses
in ascending id; a miss takes the lowest free slot, else evicts the least
recently used slot.  The pages argue that this beats placements fixed in
advance ("FreeToken：把 284B MoE 塞进游戏 PC", zhichai.net, §二, "LRU 为什么赢"
paragraph).  This module replays three placements over the same trace of
per-step routed experts, for that ablation:

* ``lru``: the library's policy (the same decisions its LRU kernel takes);
* ``prefill_static``: the n_slots experts a prefill chunk routed to most often
  (ties to the lower id) stay resident for the whole decode; a miss is fetched
  for its step only;
* ``blind_static``: experts 0 .. n_slots - 1 stay resident, chosen without any
  routing information; a miss is fetched for its step only.

Only integer bookkeeping happens here; the routing traces come from the
library's router on the GPU (``python -m routed_expert_layer_gemv_gb300.placement``).
"""
from __future__ import annotations

import json
from typing import Dict, Iterable, List, Sequence


def distinct(routed: Iterable[int]) -> List[int]:
    """The step's distinct routed experts, ascending."""
    return sorted(set(int(e) for e in routed))


class LRUCache:
    """The per-step LRU of the layer's slot table (slot_of / expert_of /
    stamps / clock), replayed on the host."""

    def __init__(self, E: int, S: int):
        self.E, self.S = E, S
        self.slot_of = [-1] * E
        self.expert_of = [-1] * S
        self.stamp = [0] * S
        self.clock = 0

    def step(self, routed: Iterable[int]) -> int:
        """Apply one step; returns its number of misses."""
        U = distinct(routed)
        hits = [e for e in U if self.slot_of[e] >= 0]
        misses = [e for e in U if self.slot_of[e] < 0]
        for e in hits:
            self.clock += 1
            self.stamp[self.slot_of[e]] = self.clock
        for e in misses:
            free = [s for s in range(self.S) if self.expert_of[s] < 0]
            s = free[0] if free else min(range(self.S), key=lambda q: (self.stamp[q], q))
            old = self.expert_of[s]
            if old >= 0:
                self.slot_of[old] = -1
            self.expert_of[s] = e
            self.slot_of[e] = s
            self.clock += 1
            self.stamp[s] = self.clock
        return len(misses)


def prefill_static_set(prefill_routed: Sequence[Sequence[int]], E: int, S: int) -> List[int]:
    """The S experts the prefill tokens routed to most often (ties to the lower id)."""
    count = [0] * E
    for row in prefill_routed:
        for e in row:
            count[int(e)] += 1
    order = sorted(range(E), key=lambda e: (-count[e], e))
    return sorted(order[:S])


def replay(trace: Sequence[Sequence[int]], E: int, S: int,
           prefill_routed: Sequence[Sequence[int]]) -> Dict[str, Dict[str, float]]:
    """Misses of each placement over the trace (one routed list per step).
    Per policy: misses, distinct (accesses), miss_rate = misses / distinct."""
    U = [distinct(step) for step in trace]
    n_distinct = sum(len(u) for u in U)
    lru = LRUCache(E, S)
    out = {"lru": sum(lru.step(u) for u in U)}
    for name, resident in (("prefill_static", set(prefill_static_set(prefill_routed, E, S))),
                           ("blind_static", set(range(min(S, E))))):
        out[name] = sum(sum(1 for e in u if e not in resident) for u in U)
    return {name: {"misses": m, "distinct": n_distinct, "miss_rate": m / max(1, n_distinct)}
            for name, m in out.items()}


def _trace(capi, torch, h, x_rows, k, max_rows):
    """Top-k ids of the library's router for the bf16 rows x_rows, routed on
    the GPU in blocks of at most max_rows rows."""
    x = torch.from_numpy(x_rows.view("int16")).view(torch.bfloat16).cuda()
    n = x.shape[0]
    idx = torch.empty(n, k, dtype=torch.int32, device="cuda")
    gates = torch.empty(n, k, dtype=torch.float32, device="cuda")
    for r0 in range(0, n, max_rows):
        r1 = min(n, r0 + max_rows)
        capi.moe_debug_router(h, x[r0:r1], r1 - r0, idx[r0:r1], gates[r0:r1])
    torch.cuda.synchronize()
    return idx.cpu().numpy()


def main() -> None:
    import argparse

    import numpy as np
    import torch

    from . import capi
    from . import workloads as wl
    from .layer import MoELayer

    ap = argparse.ArgumentParser(description="placement-policy replay over decode routing traces")
    ap.add_argument("--prefill-tokens", type=int, default=1024)
    args = ap.parse_args()
    link = None
    for work in (wl.DECODE_35B, wl.DECODE_284B):
        spec, seed = work.layer, work.seed
        rows_max = max(args.prefill_tokens, max(work.batches))
        L = MoELayer(spec, rows_max)
        W_r, b = wl.router_weights(spec, seed)
        L.set_router(W_r, b)
        xp, _ = wl.iid_tokens(seed + 1000, args.prefill_tokens, spec.d_model)
        prefill = _trace(capi, torch, L.h, xp, spec.k, rows_max)
        b_e = L.expert_bytes
        for batch in work.batches:
            xs, _ = wl.ar1_tokens(seed + batch, batch, work.steps, spec.d_model, 0.9)
            ids = _trace(capi, torch, L.h, np.ascontiguousarray(xs.reshape(-1, spec.d_model)), spec.k, rows_max)
            trace = [ids[t * batch:(t + 1) * batch].reshape(-1).tolist() for t in range(work.steps)]
            res = replay(trace, spec.E, spec.n_slots, prefill.tolist())
            if link is None:
                src = torch.empty(256 << 20, dtype=torch.uint8).pin_memory()
                dst = torch.empty_like(src, device="cuda")
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                best = None
                for _ in range(4):
                    e0.record()
                    dst.copy_(src, non_blocking=True)
                    e1.record()
                    torch.cuda.synchronize()
                    best = e0.elapsed_time(e1) if best is None else min(best, e0.elapsed_time(e1))
                link = src.numel() / (best / 1000.0) / 1e9
            for name, r in res.items():
                r["fill_MB_per_step"] = r["misses"] * b_e / work.steps / 1e6
                r["fill_us_per_step_at_link"] = r["misses"] * b_e / work.steps / (link * 1e9) * 1e6
            print(json.dumps({"workload": work.name, "batch": batch, "steps": work.steps,
                              "n_slots": spec.n_slots, "E": spec.E, "capacity": spec.n_slots / spec.E,
                              "h2d_GB_per_s": link, "prefill_tokens": args.prefill_tokens,
                              "policies": res}))
        L.close()


if __name__ == "__main__":
    main()
