"""Independent LRU models used to pin the oracle (pure Python, tiny inputs only).

Neither model is derived from the oracle's code: the oracle keeps per-slot recency
stamps and sorts; these keep explicit recency orders.
"""
from __future__ import annotations

from collections import OrderedDict


class TextbookLRU:
    """A classic single-access LRU cache of `capacity` entries (ordered dict, move to end)."""

    def __init__(self, capacity: int):
        self.capacity = capacity
        self.d: OrderedDict[int, None] = OrderedDict()

    def access(self, x: int) -> bool:
        """Returns True on a miss."""
        if x in self.d:
            self.d.move_to_end(x)
            return False
        if len(self.d) == self.capacity:
            self.d.popitem(last=False)
        self.d[x] = None
        return True

    def resident(self) -> set[int]:
        return set(self.d)


class RecencyListLRU:
    """Slot cache kept as an explicit recency list (least recent first).

    Per call: slots holding selected positions are hits; the distinct missing
    positions, smallest first, take the first non-hit slots of the list; then every
    slot used in the call goes to the back of the list, in slot-index order (they
    were all used at the same moment). Slots never used start at the front in index
    order.
    """

    def __init__(self, C: int, S: int):
        self.C, self.S = C, S
        self.order = list(range(S))       # least recently used first
        self.slot_of: dict[int, int] = {}  # position -> slot
        self.pos_in: list[int] = [-1] * S  # slot -> position
        self.touched: list[int] = [-1] * S  # call index of the slot's last use
        self.calls = 0

    def call(self, sel: list[int]):
        used = set()
        out = [-1] * len(sel)
        missing = set()
        for j, p in enumerate(sel):
            if p < 0 or p >= self.C:
                continue
            if p in self.slot_of:
                out[j] = self.slot_of[p]
                used.add(self.slot_of[p])
            else:
                missing.add(p)
        missing_sorted = sorted(missing)
        free_list = [s for s in self.order if s not in used]
        victims = free_list[: len(missing_sorted)]
        for p, s in zip(missing_sorted, victims):
            old = self.pos_in[s]
            if old >= 0:
                del self.slot_of[old]
            self.slot_of[p] = s
            self.pos_in[s] = p
            used.add(s)
        for j, p in enumerate(sel):
            if 0 <= p < self.C and out[j] < 0:
                out[j] = self.slot_of[p]
        self.order = [s for s in self.order if s not in used] + sorted(used)
        for s in used:
            self.touched[s] = self.calls
        self.calls += 1
        return out, len(missing_sorted), list(zip(missing_sorted, victims))

    def page_table(self) -> list[int]:
        pt = [-1] * self.C
        for p, s in self.slot_of.items():
            pt[p] = s
        return pt


class TextbookFIFO:
    """A classic single-access FIFO cache of `capacity` entries (a queue of arrivals;
    a hit changes nothing)."""

    def __init__(self, capacity: int):
        self.capacity = capacity
        self.q: list[int] = []

    def access(self, x: int) -> bool:
        """Returns True on a miss."""
        if x in self.q:
            return False
        if len(self.q) == self.capacity:
            self.q.pop(0)
        self.q.append(x)
        return True

    def resident(self) -> set[int]:
        return set(self.q)


_M64 = (1 << 64) - 1


def splitmix64(x: int, n: int) -> int:
    """Output number n (0, 1, ...) of SplitMix64 seeded with x, from its published
    definition (Steele, Lea and Flood 2014; Stafford's 13th mixer)."""
    z = (x + (n + 1) * 0x9E3779B97F4A7C15) & _M64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _M64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _M64
    return z ^ (z >> 31)
