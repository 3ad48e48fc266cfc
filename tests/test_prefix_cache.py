"""Host logic of the prefix-state cache (no GPU): lookup of the longest stored
prefix, block-aligned prefill pieces, LRU eviction and the slot copies it asks
the library for, checked against a fake context that records the calls and
models a slot's state as the token sequence it has consumed."""
import numpy as np
import pytest

from recurrent_decode_gb300.prefix_cache import PrefixStateCache


class FakeCtx:
    def __init__(self, n_slots):
        self.state = {s: () for s in range(n_slots)}
        self.calls = []

    def slot_copy(self, src, dst):
        self.calls.append(("copy", src, dst))
        self.state[dst] = self.state[src]

    def prefill_seq(self, slot, tokens):
        t = tuple(int(x) for x in tokens)
        self.calls.append(("prefill", slot, len(t)))
        self.state[slot] = self.state[slot] + t


def ident(a):
    return a


def admit(cache, ctx, slot, body):
    ctx.state[slot] = ()
    start = cache.restore(body, slot)
    assert ctx.state[slot] == tuple(int(x) for x in body[:start])
    cache.prefill(slot, body, start, ident)
    assert ctx.state[slot] == tuple(int(x) for x in body)  # the slot ends with the whole body consumed
    return start


def test_pieces_end_at_block_boundaries_and_states_are_stored():
    ctx = FakeCtx(4)
    cache = PrefixStateCache(ctx, [2, 3, 1], block=8)
    body = np.arange(20, dtype=np.int32)
    assert admit(cache, ctx, 0, body) == 0
    assert [c for c in ctx.calls if c[0] == "prefill"] == [("prefill", 0, 8), ("prefill", 0, 8), ("prefill", 0, 4)]
    assert len(cache) == 3 and cache.stores == 3 and cache.misses == 1
    # every stored slot holds the state after its prefix
    held = sorted(ctx.state[s] for s in (1, 2, 3))
    assert held == sorted([tuple(range(8)), tuple(range(16)), tuple(range(20))])


def test_longest_prefix_wins_and_full_body_hits():
    ctx = FakeCtx(6)
    cache = PrefixStateCache(ctx, [3, 4, 5], block=8)
    a = np.arange(20, dtype=np.int32)
    admit(cache, ctx, 0, a)
    b = np.concatenate([a[:19], [99, 98, 97]]).astype(np.int32)  # shares 19 tokens: blocks 8, 16
    assert admit(cache, ctx, 1, b) == 16
    assert admit(cache, ctx, 2, a) == 20  # identical body: the full-length entry
    assert cache.hits == 2 and cache.hit_tokens == 36
    c = np.array([5, 6, 7], np.int32)  # nothing in common
    assert admit(cache, ctx, 0, c) == 0


def test_lru_eviction_keeps_recently_used():
    ctx = FakeCtx(4)
    cache = PrefixStateCache(ctx, [2, 3], block=100)
    x = np.arange(10, dtype=np.int32)
    y = np.arange(10, 20, dtype=np.int32)
    z = np.arange(20, 30, dtype=np.int32)
    admit(cache, ctx, 0, x)       # entries: x
    admit(cache, ctx, 0, y)       # entries: x, y
    assert cache.lookup(x)[0] == 10  # touch x: y is now the oldest
    admit(cache, ctx, 0, z)       # evicts y
    assert cache.evictions == 1
    assert cache.lookup(x)[0] == 10 and cache.lookup(z)[0] == 10 and cache.lookup(y)[0] == 0
    # the evicted entry's slot was reused for z, and still holds z's state
    assert sorted(ctx.state[s] for s in (2, 3)) == sorted([tuple(range(10)), tuple(range(20, 30))])


def test_store_of_known_prefix_copies_nothing():
    ctx = FakeCtx(3)
    cache = PrefixStateCache(ctx, [1, 2], block=4)
    p = np.arange(4, dtype=np.int32)
    ctx.prefill_seq(0, p)
    cache.store(p, 0)
    n = len(ctx.calls)
    cache.store(p, 0)
    assert len(ctx.calls) == n and cache.stores == 1
    cache.store(p[:0], 0)  # empty prefix: nothing to keep
    assert len(ctx.calls) == n


def test_invalid_arguments():
    with pytest.raises(ValueError):
        PrefixStateCache(FakeCtx(1), [], block=8)
    with pytest.raises(ValueError):
        PrefixStateCache(FakeCtx(2), [1], block=0)
