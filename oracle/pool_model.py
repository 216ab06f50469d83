"""Plain model of the bounded hot-page pool's residency rules.

TEST INFRASTRUCTURE ONLY (like the rest of this package): the tests compare the
library's native planner with it; nothing in the library uses it.

It restates, as directly as possible, the reading of CFR-Atlas's resident-memory
bound (CFR-Atlas README, introduction: a byte-bounded hot cache kept across
requests, cold pages brought into reusable scratch buffers one after another and
folded; "Minimal integration": a KeepRecent { recent_tokens } policy and an
admit_regenerated_pages switch; the pages do not define either further):

* every split-KV chunk of the decode call, in (sequence, chunk) order, reads the
  logical pages that hold its keys;
* a page already in a hot slot is read there (a hit);
* a page not hot that is recent (it holds one of the sequence's last
  keep_recent_tokens keys; all pages if keep_recent_tokens < 0, none if 0) is
  admitted when admission is on and a hot slot can be had: a free one, else the one
  whose page was used longest ago (lowest slot first on ties) among pages this call
  does not read, which is evicted;
* every other page goes to a scratch slot of the pass that reads it;
* a pass takes chunks while their scratch pages fit in the scratch slots.

Linear scans everywhere; no bookkeeping beyond a list of slots.  Parity status:
pinned by hand-worked traces in ``tests/golden/pool_traces.json``.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Dict, List, Optional, Tuple


@dataclass
class Slot:
    page: Optional[int] = None   # host page held, None if free
    used: int = 0                # number of the last call that read it


@dataclass
class Pass:
    table: Dict[Tuple[int, int], int] = field(default_factory=dict)  # (b, j) -> slot
    ranges: Dict[int, Tuple[int, int]] = field(default_factory=dict)  # b -> [lo, hi)
    copies: List[Tuple[int, int]] = field(default_factory=list)       # (host page, slot)


class PoolModel:
    def __init__(self, hot_slots: int, scratch_slots: int, page_tokens: int):
        self.H, self.C, self.P = hot_slots, scratch_slots, page_tokens
        self.slots = [Slot() for _ in range(hot_slots)]
        self.calls = 0

    def slot_of(self, page: int) -> int:
        for s, sl in enumerate(self.slots):
            if sl.page == page:
                return s
        return -1

    def invalidate(self, page: int):
        s = self.slot_of(page)
        if s >= 0:
            self.slots[s] = Slot()

    def _recent(self, j: int, L: int, keep_recent: int) -> bool:
        if keep_recent < 0:
            return True
        if keep_recent == 0:
            return False
        last_key = min((j + 1) * self.P, L) - 1
        return last_key >= L - keep_recent

    def plan(self, table: List[List[int]], seq_lens: List[int], chunk: int,
             keep_recent: int = -1, admit: bool = True):
        """Returns (passes, stats) and updates the residency."""
        P = self.P
        self.calls += 1
        now = self.calls
        call_pages = []
        for b, L in enumerate(seq_lens):
            for j in range((L + P - 1) // P):
                if table[b][j] not in call_pages:
                    call_pages.append(table[b][j])
        hits = [p for p in call_pages if self.slot_of(p) >= 0]
        read_slots = {self.slot_of(p) for p in hits}
        free = [s for s in range(self.H) if s not in read_slots and self.slots[s].page is None]
        used = [s for s in range(self.H) if s not in read_slots and self.slots[s].page is not None]
        used.sort(key=lambda s: (self.slots[s].used, s))
        victims = free + used
        stats = dict(pages=len(call_pages), hits=len(hits), admitted=0, evicted=0,
                     scratch_loads=0)
        passes = [Pass()]
        scratch: List[int] = []   # pages in the current pass's scratch, in slot order
        for b, L in enumerate(seq_lens):
            for c in range((L + chunk - 1) // chunk):
                t0, t1 = c * chunk, min((c + 1) * chunk, L)
                pages = list(range(t0 // P, (t1 - 1) // P + 1))
                admitted, cold = [], []
                for j in pages:
                    hp = table[b][j]
                    if self.slot_of(hp) >= 0:
                        continue
                    if admit and self._recent(j, L, keep_recent) and victims:
                        s = victims.pop(0)
                        if self.slots[s].page is not None:
                            stats["evicted"] += 1
                        self.slots[s] = Slot(hp, now)
                        read_slots.add(s)
                        stats["admitted"] += 1
                        admitted.append((hp, s))
                    elif hp not in cold:
                        cold.append(hp)
                if len(scratch) + len([p for p in cold if p not in scratch]) > self.C:
                    passes.append(Pass())
                    scratch = []
                ps = passes[-1]
                for hp in cold:
                    if hp not in scratch:
                        scratch.append(hp)
                        ps.copies.append((hp, self.H + len(scratch) - 1))
                        stats["scratch_loads"] += 1
                ps.copies.extend(admitted)
                for j in pages:
                    hp = table[b][j]
                    s = self.slot_of(hp)
                    ps.table[(b, j)] = s if s >= 0 else self.H + scratch.index(hp)
                lo, _ = ps.ranges.get(b, (c, c))
                ps.ranges[b] = (lo, c + 1)
        for s in read_slots:
            self.slots[s].used = now
        stats["passes"] = len(passes)
        stats["copies"] = stats["admitted"] + stats["scratch_loads"]
        return passes, stats
