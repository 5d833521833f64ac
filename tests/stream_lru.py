"""Plain-Python statement of the expert cache's replacement rule (test helper).

The rule, as include/moe.h states it: each call advances a clock; every active
expert that is resident stamps its slot with the clock (a hit); the missing
experts, in increasing expert index, take the slots not stamped by this call
in increasing (stamp, slot) order (empty slots carry stamp 0), evicting the
experts held there.
"""
from __future__ import annotations


class LruModel:
    def __init__(self, n_experts: int, n_slots: int):
        self.E, self.S = n_experts, n_slots
        self.clock = 0
        self.slot_of = [-1] * n_experts
        self.expert_of = [-1] * n_slots
        self.stamp = [0] * n_slots
        self.hits = 0
        self.misses = 0

    def call(self, active: list[int]) -> list[tuple[int, int]]:
        """Apply one call's active experts; returns the (expert, slot) misses."""
        self.clock += 1
        missing = []
        for e in sorted(active):
            s = self.slot_of[e]
            if s >= 0 and self.expert_of[s] == e:
                self.stamp[s] = self.clock
                self.hits += 1
            else:
                missing.append(e)
        free = sorted((self.stamp[s], s) for s in range(self.S) if self.stamp[s] != self.clock)
        if len(missing) > len(free):
            raise ValueError("more active experts than slots")
        out = []
        for e, (_, s) in zip(missing, free):
            old = self.expert_of[s]
            if old >= 0:
                self.slot_of[old] = -1
            self.expert_of[s] = e
            self.slot_of[e] = s
            self.stamp[s] = self.clock
            out.append((e, s))
        self.misses += len(out)
        return out
