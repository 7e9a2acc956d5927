"""A second, independently written LRU residency model (test helper).

It keeps the K slots in an OrderedDict in recency order (least recently used
first) instead of per-slot ticks.  A wave touches all of its members at once:
after the wave their slots move to the most-recent end in ascending slot
order, which is what "same tick, lower slot first" means in recency-list
form.  Used only to cross-check ``oracle.lru.ResidencySim`` on exhaustive
traces.
"""

from collections import OrderedDict


class TextbookLRU:
    def __init__(self, num_experts, num_slots):
        self.E, self.K = num_experts, num_slots
        self.order = OrderedDict((s, None) for s in range(num_slots))  # slot -> expert

    def holder(self, e):
        for s, x in self.order.items():
            if x == e:
                return s
        return None

    def step(self, routed):
        """routed: iterable of expert ids. Returns list of waves, each a tuple
        (members, [(expert, slot) copied in], hits)."""
        distinct = sorted(set(routed))
        resident = [e for e in distinct if self.holder(e) is not None]
        missing = [e for e in distinct if self.holder(e) is None]
        seq = resident + missing
        out = []
        while seq:
            members, seq = seq[: self.K], seq[self.K :]
            mset = set(members)
            hits = sum(1 for e in members if self.holder(e) is not None)
            need = sorted(e for e in members if self.holder(e) is None)
            victims = [s for s, x in self.order.items() if x not in mset]
            copied = []
            for e, s in zip(need, victims):
                self.order[s] = e
                copied.append((e, s))
            touched = sorted(s for s, x in self.order.items() if x in mset)
            for s in touched:
                self.order.move_to_end(s)
            out.append((members, copied, hits))
        return out

    def resident_map(self):
        return {x: s for s, x in self.order.items() if x is not None}
