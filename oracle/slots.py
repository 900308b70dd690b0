"""The slot table's policy, stated plainly.  Test infrastructure only.

Source: goinfer, "Turn nine in under half a second":
* "How it works" -- the prompt goes to the session with the longest common
  token prefix, but only when that prefix exceeds the longest prefix the
  session has in common with any other session; the session is truncated to
  the common length and only the remaining prompt tokens are prefilled.  On
  the GPU the sessions are --kv-sessions KV slots, one conversation each; an
  unmatched prompt fills a free slot if there is one and otherwise evicts the
  slot used longest ago.
* "Use it" -- --kv-sessions 0 turns reuse off.
* "What goinfer does" / usage.prefill_reused_tokens -- the count of prompt
  tokens served from the slot instead of being prefilled.

Readings (listed in the design notes):
* R1  accept the best slot s* iff l(s*) > 0 and (threshold off or
      l(s*) > o(s*)), o(s) = longest prefix s shares with any other occupied
      slot.  With the threshold on, an accepted best slot is unique.  With it
      off, ties go to the lowest slot index.
* R1b (part of the same anti-theft rule, off with it): if accepting s* would
      cut its conversation back (l(s*) < len(s*)) while a slot is empty, the
      prompt is a new conversation and takes the empty slot.  Without this a
      second conversation that shares only the chat-template start steals the
      first one's slot whenever the table holds a single conversation, which is
      the thrash of "What we got wrong".
* R2  reused = min(l, n-1): a prompt wholly inside a slot still computes one row.
* R3  an evicted slot restarts empty.
* R4  the LRU stamp is a counter bumped whenever a slot is matched, evicted,
      written or assigned.
* n_slots == 0: one working slot, every match restarts it with reused = 0.

Parity pins (tests/test_oracle_slots.py): a brute-force reading on tiny token
alphabets; the page's turn-9 arithmetic (1922-token prompt, 1668 reused); the
thrash scenario of "What we got wrong"; the client-count shape of
"What was measured".
"""
from __future__ import annotations

from typing import List, Optional, Sequence, Tuple


def common_prefix(a: Sequence[int], b: Sequence[int]) -> int:
    n = 0
    for x, y in zip(a, b):
        if x != y:
            break
        n += 1
    return n


class SlotTable:
    def __init__(self, n_slots: int, capacity: int, threshold: bool = True):
        self.reuse = n_slots > 0
        self.n = max(n_slots, 1)
        self.cap = capacity
        self.threshold = threshold
        self.tokens: List[Optional[List[int]]] = [None] * self.n
        self.stamp = [0] * self.n
        self.clock = 0

    def _touch(self, s: int) -> None:
        self.clock += 1
        self.stamp[s] = self.clock

    def lcp_with_others(self, s: int) -> int:
        best = 0
        for t in range(self.n):
            if t != s and self.tokens[t] is not None:
                best = max(best, common_prefix(self.tokens[s], self.tokens[t]))
        return best

    def choose(self, prompt: Sequence[int]) -> Tuple[int, int, List[int]]:
        """(slot, reused, l) for a prompt, without changing the table."""
        n = len(prompt)
        l = [common_prefix(t, prompt) if t is not None else 0 for t in self.tokens]
        if self.reuse:
            best = -1
            for s in range(self.n):
                if self.tokens[s] is not None and (best < 0 or l[s] > l[best]):
                    best = s
            empty = [s for s in range(self.n) if self.tokens[s] is None]
            ok = best >= 0 and l[best] > 0
            if ok and self.threshold:
                ok = l[best] > self.lcp_with_others(best)
                if ok and empty and l[best] < len(self.tokens[best]):
                    ok = False
            if ok:
                return best, min(l[best], n - 1), l
        empty = [s for s in range(self.n) if self.tokens[s] is None]
        if empty:
            return empty[0], 0, l
        lru = min(range(self.n), key=lambda s: self.stamp[s])
        return lru, 0, l

    def match(self, prompt: Sequence[int]) -> Tuple[int, int]:
        assert len(prompt) >= 1
        s, reused, _ = self.choose(prompt)
        self.tokens[s] = list(prompt[:reused]) if reused else []
        self._touch(s)
        return s, reused

    def truncate(self, s: int, new_len: int) -> None:
        assert self.tokens[s] is not None and 0 <= new_len <= len(self.tokens[s])
        del self.tokens[s][new_len:]

    def append(self, s: int, toks: Sequence[int]) -> None:
        assert self.tokens[s] is not None and len(self.tokens[s]) + len(toks) <= self.cap
        self.tokens[s].extend(int(t) for t in toks)
        self._touch(s)

    def assign(self, s: int, toks: Sequence[int]) -> None:
        assert len(toks) <= self.cap
        self.tokens[s] = [int(t) for t in toks]
        self._touch(s)

    def length(self, s: int) -> int:
        return 0 if self.tokens[s] is None else len(self.tokens[s])

    def serve_turn(self, prompt: Sequence[int]) -> Tuple[int, int]:
        """Match, then prefill the rest: returns (slot, tokens prefilled)."""
        s, reused = self.match(prompt)
        self.append(s, prompt[reused:])
        return s, len(prompt) - reused
