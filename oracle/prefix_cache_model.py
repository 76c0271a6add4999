"""Plain model of the host prefix cache (test infrastructure, like the rest of
this package): what a match returns and which page an insert evicts, written
from the definitions, with no tree and no hashing.

Sources: "Character.AI inference optimisation" article, secret 2 (KV of every
conversation prefix kept in host memory, LRU-managed tree, longest matching
prefix also when only part of a message matches); "Character.AI best
practices" blog, "LRU cache structure"; LLM-inference workshop transcript,
01:14:28-01:16:24 (radix tree of prefixes).  Readings fixed here, the same as
the library's header: the unit is one whole page of tokens; a match is the
longest run of cached whole pages from the start; every match / insert stamps
the pages it touches with a new time; a full pool evicts the cached page that
has no cached successor (a leaf) with the oldest stamp, never one stamped by
the running insert; free slots are reused last-freed-first, slot 0 first.
"""
from __future__ import annotations


class PrefixCacheModel:
    def __init__(self, page_size: int, capacity: int):
        self.P = page_size
        self.capacity = capacity
        self.pages: dict[tuple, list] = {}  # prefix (tuple of tokens, whole pages) -> [slot, stamp]
        self.free = list(range(capacity - 1, -1, -1))
        self.clock = 0
        self.evicted = 0

    def _prefixes(self, tokens):
        n = len(tokens) // self.P
        return [tuple(tokens[: (k + 1) * self.P]) for k in range(n)]

    def match(self, tokens) -> list[int]:
        self.clock += 1
        out = []
        for pre in self._prefixes(list(tokens)):
            if pre not in self.pages:
                break
            self.pages[pre][1] = self.clock
            out.append(self.pages[pre][0])
        return out

    def _is_leaf(self, pre) -> bool:
        n = len(pre)
        return not any(len(q) == n + self.P and q[:n] == pre for q in self.pages)

    def _evict_one(self, now) -> bool:
        leaves = [(st, pre) for pre, (slot, st) in self.pages.items() if st < now and self._is_leaf(pre)]
        if not leaves:
            return False
        _, pre = min(leaves)
        self.free.append(self.pages.pop(pre)[0])
        self.evicted += 1
        return True

    def insert(self, tokens):
        """Returns [(page index, slot)] of the pages that were added."""
        self.clock += 1
        now = self.clock
        added = []
        for k, pre in enumerate(self._prefixes(list(tokens))):
            if pre in self.pages:
                self.pages[pre][1] = now
                continue
            if not self.free and not self._evict_one(now):
                break
            slot = self.free.pop()
            self.pages[pre] = [slot, now]
            added.append((k, slot))
        return added
