"""In-memory LRU of recurrent states after prompt prefixes.

An RWKV-7 sequence's whole past is its fixed-size state, so a prompt that
starts with tokens already seen can begin from the state stored after them and
prefill only the rest.  The RWKV-Runner Albatross article lists prefix-state
caching, first as an in-memory LRU, among the engine's next steps ("正在演进"
list); this is that cache for the slot pool of the C ABI.

States live in pool slots reserved for the cache (rwkv7_slot_copy moves them:
dst := src's recurrent state, dst's occurrence counts and draw counter restart).
Entries are kept at block boundaries of the prompt body (multiples of `block`
tokens from its first token) and at its full length; a lookup takes the longest
stored prefix.  With `block` equal to the library's prefill chunk
(rwkv7_prefill_seq consumes a prompt in chunks of RWKV7_MAX_STEP_BATCH tokens
counted from its first token), a body restored at a block boundary is prefilled
in exactly the chunks of an uncached run, so the results are bit-identical.

Host bookkeeping only: every computation runs in the library's kernels through
the binding (rwkv7_slot_copy, rwkv7_prefill_seq).
"""
from __future__ import annotations

import hashlib
from collections import OrderedDict

import numpy as np

from . import MAX_STEP_BATCH


def _key(tokens: np.ndarray) -> bytes:
    t = np.ascontiguousarray(tokens, dtype=np.int32)
    return hashlib.blake2b(t.tobytes(), digest_size=20).digest() + len(t).to_bytes(4, "little")


class PrefixStateCache:
    """LRU of prefix states held in the pool slots `cache_slots` of `ctx`."""

    def __init__(self, ctx, cache_slots, block: int = MAX_STEP_BATCH):
        if block <= 0:
            raise ValueError("block must be positive")
        self.ctx = ctx
        self.block = int(block)
        self.free = list(cache_slots)
        if not self.free:
            raise ValueError("the cache needs at least one slot")
        self.capacity = len(self.free)
        self.entries: OrderedDict[bytes, int] = OrderedDict()  # key -> cache slot, oldest first
        self.hits = 0
        self.misses = 0
        self.hit_tokens = 0
        self.stores = 0
        self.evictions = 0

    def __len__(self) -> int:
        return len(self.entries)

    def lookup(self, body: np.ndarray) -> tuple[int, int]:
        """(length, cache slot) of the longest stored prefix of `body`, (0, -1) if none."""
        n = len(body)
        cands = [n] + list(range((n // self.block) * self.block, 0, -self.block))
        for L in cands:
            if L <= 0:
                continue
            k = _key(body[:L])
            slot = self.entries.get(k)
            if slot is not None:
                self.entries.move_to_end(k)
                return L, slot
        return 0, -1

    def restore(self, body: np.ndarray, dst_slot: int) -> int:
        """Copy the longest stored prefix state of `body` into `dst_slot`; returns
        its length (0: nothing stored, `dst_slot` untouched)."""
        L, slot = self.lookup(body)
        if L == 0:
            self.misses += 1
            return 0
        self.ctx.slot_copy(slot, dst_slot)
        self.hits += 1
        self.hit_tokens += L
        return L

    def store(self, prefix: np.ndarray, src_slot: int) -> None:
        """Keep `src_slot`'s state as the state after `prefix` (evicting the least
        recently used entry when the cache is full)."""
        if len(prefix) == 0:
            return
        k = _key(prefix)
        if k in self.entries:
            self.entries.move_to_end(k)
            return
        if self.free:
            slot = self.free.pop()
        else:
            _, slot = self.entries.popitem(last=False)
            self.evictions += 1
        self.ctx.slot_copy(src_slot, slot)
        self.entries[k] = slot
        self.stores += 1

    def prefill(self, slot: int, body: np.ndarray, start: int, to_device) -> int:
        """Prefill body[start:] into `slot` (whose state is the state after
        body[:start]) in pieces that end at block boundaries, storing the state
        at each boundary and after the whole body.  `to_device` turns an int32
        numpy array into the device tensor rwkv7_prefill_seq takes.  Returns the
        number of tokens prefilled."""
        n = len(body)
        pos = start
        while pos < n:
            end = min(n, (pos // self.block + 1) * self.block)
            self.ctx.prefill_seq(slot, to_device(np.ascontiguousarray(body[pos:end], np.int32)))
            pos = end
            self.store(body[:pos], slot)
        return n - start
