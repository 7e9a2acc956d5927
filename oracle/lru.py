"""LRU residency simulator: waves, page-in plans, slot remap.

Follows "Paged Experts" (SGLang docs), "The K-slot table and the host
store", "A step: waves, page-in, merge" (items 1-3) and "Captured decode".
Per layer there are K GPU slots and a host copy of all E experts.  A step
takes the set of distinct experts its tokens routed to, puts the ones already
in a slot first, and cuts that order into waves of at most K.  Before a wave
runs, every expert of the wave must hold a slot: a missing one takes the slot
of the least recently used expert that is not in the wave, and its weights
are copied in.  Each routed id is then replaced by the slot of its expert.  A
decode step whose entries fit in K slots is a single wave, described by the
list of (expert, slot) copies and their count; decode and prefill steps
update the same residency state.

Readings where the pages are silent (all fixed here, and the CUDA planner
must reproduce them bit for bit):
  * start state: every slot empty (expert -1, tick 0), clock 0;
  * D = sorted distinct routed ids; R = resident members of D (ascending id),
    M = the rest (ascending id); order = R ++ M, cut into consecutive waves of
    K (R always fits in the first wave, since at most K experts are resident);
  * the clock advances once per wave; every resident member of the wave gets
    tick = clock;
  * victims are the slots whose expert is not in the wave, ordered by
    (tick, slot index) ascending, so empty slots (tick 0) go first;
  * the missing members of the wave, in ascending id, take the victims in
    that order; the victim's expert (if any) is evicted and the slot gets
    tick = clock;
  * the wave's plan is that list of (expert, slot) pairs; count = its length;
    hits = resident members of the wave; cold fills = victims that were empty.
"""

from __future__ import annotations

import dataclasses

import numpy as np


@dataclasses.dataclass
class Wave:
    experts: list[int]          # the wave's members in plan order R ++ M
    plan_expert: list[int]      # experts copied in, ascending id
    plan_slot: list[int]        # their slots
    hits: int                   # members that were already resident
    cold_fills: int             # planned slots that were empty

    @property
    def count(self) -> int:
        return len(self.plan_expert)


@dataclasses.dataclass
class StepPlan:
    waves: list[Wave]
    entry_wave: np.ndarray      # int32 [T, k]: wave holding each entry's expert
    entry_slot: np.ndarray      # int32 [T, k]: slot of each entry in that wave
    distinct: list[int]         # D

    @property
    def page_ins(self) -> int:
        return sum(w.count for w in self.waves)

    @property
    def hits(self) -> int:
        return sum(w.hits for w in self.waves)


class ResidencySim:
    """Residency state of one MoE layer's K-slot table."""

    def __init__(self, num_experts: int, num_slots: int):
        if not 1 <= num_slots <= num_experts:
            raise ValueError("need 1 <= K <= E")
        self.E = num_experts
        self.K = num_slots
        self.reset()

    def reset(self) -> None:
        self.slot_expert = [-1] * self.K
        self.slot_tick = [0] * self.K
        self.expert_slot = [-1] * self.E
        self.clock = 0

    def resident(self, e: int) -> bool:
        return self.expert_slot[e] >= 0

    def check_invariants(self) -> None:
        for s, e in enumerate(self.slot_expert):
            if e >= 0:
                assert self.expert_slot[e] == s
        for e, s in enumerate(self.expert_slot):
            if s >= 0:
                assert self.slot_expert[s] == e

    def step(self, ids: np.ndarray) -> StepPlan:
        """Plan one layer step for routed ids (int [T, k]) and update state."""
        ids = np.asarray(ids)
        distinct = sorted(set(int(e) for e in ids.reshape(-1)))
        if distinct and not (0 <= distinct[0] and distinct[-1] < self.E):
            raise ValueError("expert id out of range")
        R = [e for e in distinct if self.resident(e)]
        M = [e for e in distinct if not self.resident(e)]
        order = R + M
        waves: list[Wave] = []
        wave_of = {}
        slot_in_wave = {}
        for w0 in range(0, len(order), self.K):
            members = order[w0 : w0 + self.K]
            mset = set(members)
            self.clock += 1
            hits = 0
            for e in members:
                if self.resident(e):
                    self.slot_tick[self.expert_slot[e]] = self.clock
                    hits += 1
            victims = sorted(
                (s for s in range(self.K) if self.slot_expert[s] not in mset),
                key=lambda s: (self.slot_tick[s], s),
            )
            missing = sorted(e for e in members if not self.resident(e))
            plan_e, plan_s, cold = [], [], 0
            for e, s in zip(missing, victims):
                old = self.slot_expert[s]
                if old >= 0:
                    self.expert_slot[old] = -1
                else:
                    cold += 1
                self.slot_expert[s] = e
                self.expert_slot[e] = s
                self.slot_tick[s] = self.clock
                plan_e.append(e)
                plan_s.append(s)
            for e in members:
                wave_of[e] = len(waves)
                slot_in_wave[e] = self.expert_slot[e]
            waves.append(Wave(members, plan_e, plan_s, hits, cold))
        flat = ids.reshape(-1)
        entry_wave = np.array([wave_of[int(e)] for e in flat], np.int32).reshape(ids.shape)
        entry_slot = np.array([slot_in_wave[int(e)] for e in flat], np.int32).reshape(ids.shape)
        return StepPlan(waves, entry_wave, entry_slot, distinct)
