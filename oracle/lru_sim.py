"""Pure-Python replay of the expert slot pool (LRU) — TEST INFRASTRUCTURE ONLY.

Follows page 4 ("llama.cpp MoE缓存实测", section "MoE缓存到底缓存了什么"):
one VRAM slot pool per type/shape group, shared by all layers of the group,
hits read the slot, misses are uploaded, eviction is least-recently-used; and
page 1 (section 3.2): the victim is the least-recently-used expert that is not
part of the current request.

Rules, per ``ensure(layer, ids)`` on one group:
  1. the request is the set of distinct expert ids, taken in ascending order;
  2. more distinct ids than slots is an error (capacity);
  3. hits first, in ascending id order, each stamped with ++clock;
  4. then misses, in ascending id order: the lowest-numbered free slot, else the
     slot with the smallest stamp whose owner is not in this request; the new
     owner is stamped with ++clock.
One query is counted per distinct (layer, expert) per call.
"""
from __future__ import annotations

from typing import Dict, Iterable, List, Optional, Tuple


class CapacityError(Exception):
    pass


class LRUSim:
    def __init__(self, n_slots: int):
        if n_slots <= 0:
            raise ValueError("n_slots must be positive")
        self.n_slots = n_slots
        self.owner: List[Optional[Tuple[int, int]]] = [None] * n_slots
        self.stamp: List[int] = [0] * n_slots
        self.where: Dict[Tuple[int, int], int] = {}
        self.clock = 0
        self.hits = 0
        self.misses = 0
        self.evictions = 0

    def ensure(self, layer: int, ids: Iterable[int]) -> Tuple[Dict[int, int], List[int], List[int]]:
        """Returns ({expert: slot}, hit ids, miss ids) for one request."""
        req = sorted(set(int(e) for e in ids))
        if len(req) > self.n_slots:
            raise CapacityError(f"{len(req)} distinct experts > {self.n_slots} slots")
        keys = {(layer, e) for e in req}
        result: Dict[int, int] = {}
        hit_ids = [e for e in req if (layer, e) in self.where]
        miss_ids = [e for e in req if (layer, e) not in self.where]
        for e in hit_ids:
            s = self.where[(layer, e)]
            self.clock += 1
            self.stamp[s] = self.clock
            result[e] = s
        for e in miss_ids:
            free = [s for s in range(self.n_slots) if self.owner[s] is None]
            if free:
                s = free[0]
            else:
                cands = [s for s in range(self.n_slots) if self.owner[s] not in keys]
                s = min(cands, key=lambda i: self.stamp[i])
                del self.where[self.owner[s]]
                self.evictions += 1
            self.owner[s] = (layer, e)
            self.where[(layer, e)] = s
            self.clock += 1
            self.stamp[s] = self.clock
            result[e] = s
        self.hits += len(hit_ids)
        self.misses += len(miss_ids)
        return result, hit_ids, miss_ids


def slots_for_budget(budget_bytes: int, per_expert_bytes: Iterable[int], k: int) -> List[int]:
    """Slot count per group from a byte budget (page 4, "配置之前，先算清楚你的专家有多大").

    Reading: every group gets the same slot count N, the largest N with
    N * sum(per-expert bytes of each group) <= budget; a group with fewer than
    k + 1 slots (one token's k experts plus one to evict) is under budget.
    Returns [] if every group is under budget (the refusal case).
    """
    per = list(per_expert_bytes)
    n = budget_bytes // sum(per)
    if n < k + 1:
        return []
    return [n] * len(per)
