"""Reference model of the decode-time expert cache (LRU over device slots).

TEST INFRASTRUCTURE.  Only the test suite, the smoke check in
``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` may import this
module.  It shares no code with the library.

The pages flag expert caching as an optimisation that the routing analysis
makes attractive (paper-graph-ui summary, "Expert caching hint" and the
Table 5 discussion of temporal locality: consecutive tokens often reuse the
same experts, so frequently used experts can stay in GPU memory while the
rest live in CPU memory, cutting host-to-device transfers).  They give no
policy, so this library's is written out plainly:

  * C device slots, each holding one expert's three weight blocks.
  * Per step, the set N of experts that the step's tokens were routed to.
  * Every expert of N that is resident is a hit; every other one a miss, loaded
    into a slot, misses taken in increasing expert index.
  * A miss takes the lowest-index empty slot if there is one; otherwise it
    evicts the least recently used resident expert that is not in N (least
    recent = smallest step of last use; ties to the lowest slot index).
  * Every expert of N gets its slot's last-use step set to the current step,
    then the step counter advances.
  * |N| > C is an error (the step cannot hold its experts at once).
"""
from __future__ import annotations

from dataclasses import dataclass, field


class CacheTooSmall(ValueError):
    pass


@dataclass
class LRUCache:
    E: int
    C: int
    slot_of: list = field(default_factory=list)    # expert -> slot or -1
    expert_in: list = field(default_factory=list)  # slot -> expert or -1
    last_use: list = field(default_factory=list)   # slot -> step of last use (-1: never)
    step: int = 0
    hits: int = 0
    misses: int = 0

    def __post_init__(self):
        if not (1 <= self.C <= self.E):
            raise ValueError("need 1 <= C <= E")
        self.slot_of = [-1] * self.E
        self.expert_in = [-1] * self.C
        self.last_use = [-1] * self.C

    def plan(self, needed):
        """needed: iterable of expert indices.  Returns the loads
        [(expert, slot), ...] in the order they are made."""
        need = sorted(set(int(e) for e in needed))
        if any(e < 0 or e >= self.E for e in need):
            raise ValueError("expert index out of range")
        if len(need) > self.C:
            raise CacheTooSmall(f"{len(need)} experts needed, {self.C} slots")
        need_set = set(need)
        loads = []
        for e in need:
            if self.slot_of[e] >= 0:
                self.hits += 1
                continue
            self.misses += 1
            empty = [s for s in range(self.C) if self.expert_in[s] < 0]
            if empty:
                s = empty[0]
            else:
                s = self.victim([s for s in range(self.C) if self.expert_in[s] not in need_set])
                self.slot_of[self.expert_in[s]] = -1
            self.expert_in[s] = e
            self.slot_of[e] = s
            loads.append((e, s))
        loaded = {e for e, _ in loads}
        for e in need:
            self.touch(self.slot_of[e], e in loaded)
        self.step += 1
        return loads

    def victim(self, candidates):
        """The slot to evict: least recently used, ties to the lowest index."""
        return min(candidates, key=lambda s: (self.last_use[s], s))

    def touch(self, slot, loaded_now: bool):
        """Mark the slot's expert as used at the current step."""
        self.last_use[slot] = self.step


def simulate(trace, E: int, C: int):
    """Run the policy over a trace of per-step needed-expert sets; returns the
    cache and the list of per-step loads."""
    c = LRUCache(E, C)
    return c, [c.plan(n) for n in trace]
