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

Policy variants (each off by default; with both off the rules above are unchanged):
  * admit_after = theta (frequency admission; page 3, section "2.2 第二层专家缓存层": count
    each expert's accesses and move it into VRAM once the count passes a threshold):
    every request counts one access per distinct (layer, expert); a miss whose count,
    this access included, is below theta is "bypassed" — served from host memory, no slot,
    no LRU change — and still counted as a miss; from theta on it is admitted by rule 4.
    theta = 1 is plain LRU.  The capacity check counts hits plus admitted misses only.
  * window = W tokens (page 1, section "4.3 运行时配置bat脚本里的魔鬼参数": an expert not
    used within the last W tokens is unloaded): the pool keeps a token clock, advanced by
    the ubatch's token count at every request of the group's first layer; before a
    request, every slot whose last use is more than W tokens behind the clock is freed
    (its expert becomes non-resident), then rules 1-4 apply.

Speculative requests (cross-layer prefetch; page 3, section "2.3 第三层传输与计算重叠层":
the experts the next one or two layers will use are prefetched while the current layer
computes): ``prefetch(layer, ids)`` applies rules 1-4 to the predicted ids like a request
(hits stamped, misses given slots — under admission the misses the real access would
admit — without counting an access), with its own statistics, and is abandoned — nothing
changes — when it needs more slots than the pool has or would evict a slot of the last
real request (that layer's work may still be using it).
"""
from __future__ import annotations

from typing import Dict, Iterable, List, Optional, Tuple


class CapacityError(Exception):
    pass


class LRUSim:
    def __init__(self, n_slots: int, admit_after: int = 1, window: int = 0, first_layer: int = 0):
        if n_slots <= 0:
            raise ValueError("n_slots must be positive")
        if admit_after < 1 or window < 0:
            raise ValueError("admit_after >= 1 and window >= 0")
        self.n_slots = n_slots
        self.admit_after = admit_after
        self.window = window
        self.first_layer = first_layer
        self.owner: List[Optional[Tuple[int, int]]] = [None] * n_slots
        self.stamp: List[int] = [0] * n_slots
        self.last_tok: List[int] = [0] * n_slots
        self.where: Dict[Tuple[int, int], int] = {}
        self.count: Dict[Tuple[int, int], int] = {}
        self.clock = 0
        self.tok = 0
        self.hits = 0
        self.misses = 0
        self.evictions = 0
        self.bypassed = 0
        self.window_evictions = 0
        self.last_real_slots: set = set()
        self.pf_queries = 0
        self.pf_hits = 0
        self.pf_fills = 0
        self.pf_aborts = 0

    def ensure(self, layer: int, ids: Iterable[int], n_tokens: int = 1
               ) -> Tuple[Dict[int, int], List[int], List[int]]:
        """Returns ({expert: slot, -1 if bypassed}, hit ids, miss ids) for one request."""
        req = sorted(set(int(e) for e in ids))
        if layer == self.first_layer:
            tok = self.tok + n_tokens
        else:
            tok = self.tok
        keys = {(layer, e) for e in req}
        # the window: slots unused for more than W tokens are freed first
        stale = []
        if self.window > 0:
            stale = [s for s in range(self.n_slots)
                     if self.owner[s] is not None and tok - self.last_tok[s] > self.window]
        resident = lambda e: (layer, e) in self.where and self.where[(layer, e)] not in stale
        hit_ids = [e for e in req if resident(e)]
        miss_ids = [e for e in req if not resident(e)]
        counts = {e: self.count.get((layer, e), 0) + 1 for e in req}
        admitted = [e for e in miss_ids if counts[e] >= self.admit_after]
        bypass = [e for e in miss_ids if counts[e] < self.admit_after]
        if len(hit_ids) + len(admitted) > self.n_slots:
            raise CapacityError(f"{len(hit_ids) + len(admitted)} experts need slots > {self.n_slots} slots")
        # commit
        self.tok = tok
        for s in stale:
            del self.where[self.owner[s]]
            self.owner[s] = None
            self.window_evictions += 1
        for e in req:
            self.count[(layer, e)] = counts[e]
        result: Dict[int, int] = {}
        for e in hit_ids:
            s = self.where[(layer, e)]
            self.clock += 1
            self.stamp[s] = self.clock
            self.last_tok[s] = tok
            result[e] = s
        for e in admitted:
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
            self.last_tok[s] = tok
            result[e] = s
        for e in bypass:
            result[e] = -1
        self.hits += len(hit_ids)
        self.misses += len(miss_ids)
        self.bypassed += len(bypass)
        self.last_real_slots = {s for s in result.values() if s >= 0}
        return result, hit_ids, miss_ids

    def prefetch(self, layer: int, ids: Iterable[int]) -> Dict[int, int]:
        """A speculative request; returns {expert: slot, -1 if not resident} ({} if abandoned)."""
        req = sorted(set(int(e) for e in ids))
        keys = {(layer, e) for e in req}
        hit_ids = [e for e in req if (layer, e) in self.where]
        miss_ids = [e for e in req if (layer, e) not in self.where]
        # what the real access would admit (count + 1 >= theta), without counting the access
        admitted = [e for e in miss_ids if self.count.get((layer, e), 0) + 1 >= self.admit_after]
        if len(hit_ids) + len(admitted) > self.n_slots:
            self.pf_aborts += 1
            return {}
        # the victims the misses would take (after the free slots), oldest first
        n_free = sum(1 for s in range(self.n_slots) if self.owner[s] is None)
        n_evict = max(0, len(admitted) - n_free)
        cands = sorted((s for s in range(self.n_slots) if self.owner[s] not in keys and self.owner[s] is not None),
                       key=lambda i: self.stamp[i])
        if any(s in self.last_real_slots for s in cands[:n_evict]):
            self.pf_aborts += 1
            return {}
        result: Dict[int, int] = {}
        for e in hit_ids:
            s = self.where[(layer, e)]
            self.clock += 1
            self.stamp[s] = self.clock
            result[e] = s
        for e in admitted:
            free = [s for s in range(self.n_slots) if self.owner[s] is None]
            if free:
                s = free[0]
            else:
                s = min((s for s in range(self.n_slots) if self.owner[s] not in keys), key=lambda i: self.stamp[i])
                del self.where[self.owner[s]]
                self.evictions += 1
            self.owner[s] = (layer, e)
            self.where[(layer, e)] = s
            self.clock += 1
            self.stamp[s] = self.clock
            result[e] = s
        for e in miss_ids:
            result.setdefault(e, -1)
        self.pf_queries += len(req)
        self.pf_hits += len(hit_ids)
        self.pf_fills += len(admitted)
        return result


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
