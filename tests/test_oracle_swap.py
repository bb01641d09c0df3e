"""Pins for swap-out / swap-in (preemption to a CPU pool, aiqz.cc "vLLM PagedAttention
engine", section 连续批处理：随到随走的新秩序): hand-worked walk-throughs of the FIFO
rules, per-pool conservation under random operation sequences, the logical content of
every sequence (and the decode oracle's output) unchanged by a round trip, and planted
mistakes that a pin has to catch."""
import random

import numpy as np
import pytest

import workloads
from oracle import attention, cache_ops, formats, sizing
from oracle.block_pool import BlockPool, PoolExhausted, UnknownSequence, WrongTier


def test_walkthrough_one_sequence():
    # 8 device blocks and 4 CPU blocks, both free lists in id order, B = 16.
    pool = BlockPool(8, 16, num_cpu_blocks=4)
    pool.allocate("A", 40)                   # blocks 0, 1, 2
    pool.allocate("B", 20)                   # blocks 3, 4
    assert pool.swap_out(["A"]) == [(0, 0), (1, 1), (2, 2)]
    assert pool.is_swapped("A") and not pool.is_swapped("B")
    assert pool.block_table("A") == [0, 1, 2]            # CPU ids now
    assert pool.free_list == [5, 6, 7, 0, 1, 2]          # returned to the tail, in order
    assert pool.cpu_free_list == [3]
    pool.allocate("C", 17)                   # takes 5, 6 from the head
    assert pool.swap_in(["A"]) == [(0, 7), (1, 0), (2, 1)]
    assert pool.block_table("A") == [7, 0, 1] and not pool.is_swapped("A")
    assert pool.free_list == [2] and pool.cpu_free_list == [3, 0, 1, 2]
    assert pool.context_len("A") == 40


def test_walkthrough_shared_blocks():
    pool = BlockPool(8, 16, num_cpu_blocks=8)
    pool.allocate("P", 40)                   # 0, 1, 2 (last block partly filled)
    pool.fork("P", "Q")                      # Q shares 0, 1, 2
    slot, cow = pool.append_slot("Q")        # Q copies its shared partial block 2 -> 3
    assert cow == (2, 3) and slot == 3 * 16 + 8
    # Q alone: its blocks 0 and 1 are still held by P, so they stay on the device
    assert pool.swap_out(["Q"]) == [(0, 0), (1, 1), (3, 2)]
    assert pool.refcount[0] == 1 and pool.refcount[1] == 1 and pool.refcount[3] == 0
    assert pool.free_list == [4, 5, 6, 7, 3]
    assert pool.cpu_refcount[:3] == [1, 1, 1]
    pool.free("Q")                           # a swapped sequence frees its CPU blocks
    assert pool.cpu_free_list == [3, 4, 5, 6, 7, 0, 1, 2]
    # P and a fork of it together: each distinct block once, carrying both references
    pool.fork("P", "R")
    assert pool.swap_out(["P", "R"]) == [(0, 3), (1, 4), (2, 5)]
    assert pool.cpu_refcount[3:6] == [2, 2, 2]
    assert pool.free_list == [4, 5, 6, 7, 3, 0, 1, 2]
    assert pool.swap_in(["R"]) == [(3, 4), (4, 5), (5, 6)]
    assert pool.cpu_refcount[3:6] == [1, 1, 1] and pool.refcount[4:7] == [1, 1, 1]


def test_errors_change_nothing():
    pool = BlockPool(4, 16, num_cpu_blocks=2)
    pool.allocate(0, 40)                     # 3 blocks
    pool.allocate(1, 1)
    before = (list(pool.free_list), list(pool.cpu_free_list), dict(pool.tables))
    with pytest.raises(PoolExhausted):
        pool.swap_out([0])                   # needs 3 CPU blocks, 2 free
    assert (pool.free_list, pool.cpu_free_list, pool.tables) == before
    assert not pool.is_swapped(0)
    with pytest.raises(WrongTier):
        pool.swap_in([1])                    # resident
    with pytest.raises(UnknownSequence):
        pool.swap_out([7])
    with pytest.raises(ValueError):
        pool.swap_out([1, 1])
    pool.swap_out([1])
    with pytest.raises(WrongTier):
        pool.append_slot(1)
    with pytest.raises(WrongTier):
        pool.fork(1, 2)
    with pytest.raises(WrongTier):
        pool.swap_out([1])
    pool.free(0)
    pool.allocate(3, 64)                     # all 4 device blocks
    with pytest.raises(PoolExhausted):
        pool.swap_in([1])
    assert pool.is_swapped(1)


def check_tiers(pool):
    """Conservation in each pool: every block is free or referenced, never both, and its
    reference count is the number of table entries naming it."""
    for on_cpu, n, ref, free in ((False, pool.num_blocks, pool.refcount, pool.free_list),
                                 (True, pool.num_cpu_blocks, pool.cpu_refcount,
                                  pool.cpu_free_list)):
        tables = [t for s, t in pool.tables.items() if (s in pool.swapped) == on_cpu]
        live = set(b for t in tables for b in t)
        assert len(live) + len(free) == n and not live & set(free)
        assert len(set(free)) == len(free)
        for b in range(n):
            assert ref[b] == sum(t.count(b) for t in tables)
    for seq, table in pool.tables.items():
        assert len(table) == sizing.blocks_needed(pool.ctx[seq], pool.block_size)


def random_ops(pool, rng, steps, on_cow=None, on_swap=None):
    for _ in range(steps):
        next_id = max([s for s in pool.tables if isinstance(s, int)] + [999]) + 1
        live = [s for s in pool.tables if s not in pool.swapped]
        out = sorted(pool.swapped)
        op = rng.random()
        try:
            if op < 0.2 or not pool.tables:
                pool.allocate(next_id, rng.randint(0, 9))
            elif op < 0.45 and live:
                seq = rng.choice(live)
                slot, cow = pool.append_slot(seq)
                if on_cow:
                    on_cow(seq, slot, cow)
            elif op < 0.55 and live:
                pool.fork(rng.choice(live), next_id)
            elif op < 0.7 and live:
                group = rng.sample(live, rng.randint(1, min(3, len(live))))
                pairs = pool.swap_out(group)
                if on_swap:
                    on_swap(True, pairs)
            elif op < 0.85 and out:
                group = rng.sample(out, rng.randint(1, min(3, len(out))))
                pairs = pool.swap_in(group)
                if on_swap:
                    on_swap(False, pairs)
            else:
                pool.free(rng.choice(list(pool.tables)))
        except PoolExhausted:
            pass
        check_tiers(pool)


def test_random_operations_keep_both_pools_consistent():
    rng = random.Random(7)
    for _ in range(150):
        pool = BlockPool(16, rng.choice([1, 2, 4]), rng.sample(range(16), 16),
                         num_cpu_blocks=rng.choice([4, 12]),
                         cpu_free_order=None)
        random_ops(pool, rng, 60)


class Caches:
    """A device pool and a CPU pool of K/V blocks driven by the bookkeeping: every token
    written gets a distinct value; copies follow copy_blocks and swap_blocks."""

    def __init__(self, pool, hkv=2, d=4):
        self.pool = pool
        shape = (pool.num_blocks, hkv, pool.block_size, d)
        cshape = (pool.num_cpu_blocks, hkv, pool.block_size, d)
        self.k, self.v = np.zeros(shape, np.uint16), np.zeros(shape, np.uint16)
        self.ck, self.cv = np.zeros(cshape, np.uint16), np.zeros(cshape, np.uint16)
        self.logical = {}                    # seq -> list of (k row, v row) by position
        self.counter = 1

    def row(self):
        hkv, d = self.k.shape[1], self.k.shape[3]
        r = np.arange(self.counter, self.counter + hkv * d, dtype=np.uint16).reshape(hkv, d)
        self.counter += hkv * d
        return r

    def on_cow(self, seq, slot, cow):
        if cow is not None:
            self.k, self.v = cache_ops.copy_blocks(self.k, self.v, [cow])
        k, v = self.row(), self.row() + 7
        self.k, self.v = cache_ops.reshape_and_cache(self.k, self.v, k[None], v[None],
                                                     np.array([slot]))

    def on_swap(self, out, pairs):
        if not pairs:
            return
        if out:
            self.ck, self.cv = cache_ops.swap_blocks(self.k, self.v, self.ck, self.cv, pairs)
        else:
            self.k, self.v = cache_ops.swap_blocks(self.ck, self.cv, self.k, self.v, pairs)

    def contents(self, seq):
        pool = self.pool
        k, v = (self.ck, self.cv) if pool.is_swapped(seq) else (self.k, self.v)
        t = pool.block_table(seq)
        B = pool.block_size
        return [(k[t[i // B], :, i % B].copy(), v[t[i // B], :, i % B].copy())
                for i in range(pool.context_len(seq))]


def test_round_trips_keep_every_sequence_content():
    """Every sequence reads the same rows at every position whatever the swaps did: a
    wrong pair, a missed block or a block freed too early changes some row."""
    rng = random.Random(11)
    for trial in range(40):
        pool = BlockPool(24, rng.choice([2, 4]), rng.sample(range(24), 24), num_cpu_blocks=16,
                         cpu_free_order=rng.sample(range(16), 16))
        c = Caches(pool)
        for _ in range(80):
            before = {s: c.contents(s) for s in pool.tables}
            random_ops(pool, rng, 1, on_cow=c.on_cow, on_swap=c.on_swap)
            for s in pool.tables:
                if s in before:
                    now = c.contents(s)
                    # a grown sequence keeps its old rows; others are unchanged
                    assert len(now) >= len(before[s])
                    for (k0, v0), (k1, v1) in zip(before[s], now):
                        assert np.array_equal(k0, k1) and np.array_equal(v0, v1)


def test_decode_after_a_round_trip_is_unchanged():
    """The decode oracle over the swapped-in tables equals the decode before the swap,
    bit for bit: the blocks moved, the logical sequences did not."""
    wl = workloads.tiny()
    B = wl.block_size
    pool = BlockPool(wl.num_blocks, B, wl.free_order, num_cpu_blocks=wl.num_blocks)
    shape = (wl.num_blocks, wl.num_kv_heads, B, wl.head_dim)
    nan = formats.FORMATS[wl.dtype]["qnan"]
    kc, vc = np.full(shape, nan, np.uint16), np.full(shape, nan, np.uint16)
    slots = []
    for s in range(wl.num_seqs):
        pool.allocate(s, int(wl.context_lens[s]))
        slots += [pool.slot(s, t) for t in range(int(wl.context_lens[s]))]
    kc, vc = cache_ops.reshape_and_cache(kc, vc, wl.keys, wl.values, np.array(slots))

    def tables():
        t = np.full((wl.num_seqs, wl.max_blocks_per_seq), -1, np.int32)
        for s in range(wl.num_seqs):
            row = pool.block_table(s)
            t[s, :len(row)] = row
        return t
    t_before = tables()
    before, err = attention.paged_decode(wl.q, kc, vc, t_before, wl.context_lens, wl.scale, B,
                                         wl.dtype)
    assert not err.any()
    ck, cv = np.full(shape, nan, np.uint16), np.full(shape, nan, np.uint16)
    ck, cv = cache_ops.swap_blocks(kc, vc, ck, cv, pool.swap_out([1, 3]))
    pool.allocate(99, 40)                    # someone else takes freed device blocks
    kc, vc = cache_ops.swap_blocks(ck, cv, kc, vc, pool.swap_in([3, 1]))
    after, err = attention.paged_decode(wl.q, kc, vc, tables(), wl.context_lens, wl.scale, B,
                                        wl.dtype)
    assert not err.any()
    np.testing.assert_array_equal(before, after)
    assert (tables()[[1, 3]] != t_before[[1, 3]]).any()  # the blocks did move


def test_planted_mistakes_are_caught():
    """(1) A swap that copies a shared block once per referencing sequence takes more CPU
    blocks than the distinct-block count; (2) a swap_in that returns pairs reversed breaks
    the content check; (3) a swap that frees a block still held elsewhere breaks
    conservation."""
    class NoDedup(BlockPool):
        def swap_out(self, seqs):
            pairs = []
            for s in seqs:
                pairs += super().swap_out([s])
            return pairs
    pool = NoDedup(8, 16, num_cpu_blocks=8)
    pool.allocate("P", 20)
    pool.fork("P", "R")
    pool.swap_out(["P", "R"])
    assert 8 - len(pool.cpu_free_list) != 2      # the correct pool takes 2 CPU blocks

    pool = BlockPool(8, 4, num_cpu_blocks=8)
    c = Caches(pool)
    pool.allocate("A", 0)
    for _ in range(10):
        c.on_cow("A", *pool.append_slot("A"))
    want = c.contents("A")
    c.on_swap(True, pool.swap_out(["A"]))
    c.on_swap(False, [(d, s) for s, d in pool.swap_in(["A"])])
    got = c.contents("A")
    assert any(not np.array_equal(a[0], b[0]) for a, b in zip(want, got))

    class EagerFree(BlockPool):
        def swap_out(self, seqs):
            pairs = super().swap_out(seqs)
            for b, _ in pairs:
                if self.refcount[b] > 0 and b not in self.free_list:
                    self.refcount[b] = 0
                    self.free_list.append(b)
            return pairs
    pool = EagerFree(8, 16, num_cpu_blocks=8)
    pool.allocate("P", 20)
    pool.fork("P", "Q")
    pool.swap_out(["Q"])
    with pytest.raises(AssertionError):
        check_tiers(pool)
