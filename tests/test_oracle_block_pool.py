"""Pins for the oracle's block bookkeeping: the allocator demo walk-through the pages
print, the allocation policy, copy-on-write counts in closed form, and invariants under
random operation sequences on a small pool."""
import random

import pytest

from oracle import sizing
from oracle.block_pool import BlockPool, PoolExhausted, UnknownSequence


def test_allocator_demo_walkthrough(golden):
    g = golden("allocator_demo.json")
    pool = BlockPool(g["num_blocks"], g["block_size"])
    for rid, n in g["requests"]:
        pool.allocate(rid, n)
    for rid, table in g["tables_after_abc"].items():
        assert pool.block_table(rid) == table
    assert pool.free_list == g["free_after_abc"]
    pool.free("A")
    pool.free("C")
    assert pool.num_free() == g["free_count_after_freeing_a_and_c"]
    rid, n = g["request_d"]
    pool.allocate(rid, n)
    assert pool.block_table(rid) == g["table_d"]
    # utilisation of D counted over allocated tokens: 6 of 8 slots
    assert sizing.effective_utilisation([pool.context_len("D")],
                                        [len(pool.block_table("D")) * g["block_size"]]) == 0.75


def test_allocation_policy():
    # horeb.top, section 分配策略: prefill ceil(prompt/16) blocks; decode adds a block every
    # 16 tokens; a finished sequence returns every block.
    pool = BlockPool(64, 16)
    pool.allocate(0, 37)
    assert len(pool.block_table(0)) == 3
    for _ in range(11):                      # 37 -> 48 tokens: still 3 blocks
        pool.append_slot(0)
    assert len(pool.block_table(0)) == 3
    pool.append_slot(0)                      # token 48 opens block 4
    assert len(pool.block_table(0)) == 4
    for _ in range(15):
        pool.append_slot(0)
    assert len(pool.block_table(0)) == 4 and pool.context_len(0) == 64
    pool.free(0)
    assert pool.num_free() == 64


def test_append_slot_addresses_follow_the_table():
    pool = BlockPool(32, 8, initial_free_order=list(range(31, -1, -1)))
    pool.allocate(7, 0)
    slots = [pool.append_slot(7)[0] for _ in range(20)]
    table = pool.block_table(7)
    assert table == [31, 30, 29]
    assert slots == [table[t // 8] * 8 + t % 8 for t in range(20)]


def test_exhaustion_rejects_without_change():
    # daiw.org, section 速查卡 运维提示: an exhausted pool rejects new requests.
    pool = BlockPool(4, 16)
    pool.allocate(0, 40)                     # 3 blocks
    before = (list(pool.free_list), pool.block_table(0), list(pool.refcount))
    with pytest.raises(PoolExhausted):
        pool.allocate(1, 33)                 # needs 3, one free
    assert 1 not in pool.tables
    assert (list(pool.free_list), pool.block_table(0), list(pool.refcount)) == before
    pool.allocate(1, 16)                     # takes the last block
    with pytest.raises(PoolExhausted):
        pool.append_slot(1)                  # token 16 needs a new block
    assert pool.context_len(1) == 16 and len(pool.block_table(1)) == 1


def test_unknown_and_duplicate_sequences():
    pool = BlockPool(8, 4)
    with pytest.raises(UnknownSequence):
        pool.free(3)
    with pytest.raises(UnknownSequence):
        pool.append_slot(3)
    pool.allocate(3, 1)
    with pytest.raises(UnknownSequence):
        pool.allocate(3, 1)
    with pytest.raises(UnknownSequence):
        pool.fork(3, 3)


def test_fork_shares_and_cow_copies_only_the_partial_last_block():
    pool = BlockPool(16, 4)
    pool.allocate("p", 6)                    # blocks [0, 1], last holds 2 tokens
    pool.fork("p", "c")
    assert pool.block_table("c") == [0, 1]
    assert pool.refcount[0] == pool.refcount[1] == 2
    slot, cow = pool.append_slot("c")        # writes into the shared partial block
    assert cow == (1, 2)
    assert pool.block_table("c") == [0, 2] and pool.block_table("p") == [0, 1]
    assert slot == 2 * 4 + 2
    assert pool.refcount[1] == 1 and pool.refcount[2] == 1 and pool.refcount[0] == 2
    slot, cow = pool.append_slot("p")        # parent is now the sole owner: in place
    assert cow is None and slot == 1 * 4 + 2
    pool.free("p")
    assert pool.free_list[-1] == 1           # block 0 still referenced by "c"
    pool.free("c")
    assert sorted(pool.free_list) == list(range(16))


def test_full_shared_blocks_stay_shared():
    pool = BlockPool(16, 4)
    pool.allocate("p", 8)                    # two full blocks
    pool.fork("p", "c")
    _, cow = pool.append_slot("c")           # token 8 opens a fresh block, no copy
    assert cow is None
    assert pool.block_table("c")[:2] == pool.block_table("p")


def beam_script(pool, prompts=2, beams=8, prefix=1024, private=None):
    """The shared-prefix beam workload: each prompt holds prefix + 1 generated tokens,
    forks into ``beams`` beams, then each beam writes its private tokens."""
    cows = []
    for p in range(prompts):
        root = p * beams
        pool.allocate(root, prefix)
        pool.append_slot(root)               # the shared first generated token
        for b in range(1, beams):
            pool.fork(root, root + b)
    for p in range(prompts):
        for b in range(beams):
            seq = p * beams + b
            for _ in range(private[seq]):
                _, cow = pool.append_slot(seq)
                if cow:
                    cows.append(cow)
    return cows


def test_beam_workload_closed_form():
    # 1024 = 64 full blocks; the 1025th token makes a shared partial 65th block with
    # refcount 8.  The first 7 beams to write copy it, the 8th writes in place: 7 copies
    # per prompt, 2*64 shared + 16 distinct last blocks.
    rng = random.Random(0)
    private = [rng.randint(1, 15) for _ in range(16)]
    pool = BlockPool(256, 16)
    cows = beam_script(pool, private=private)
    assert len(cows) == 14
    used = 256 - pool.num_free()
    assert used == 2 * 64 + 16
    for seq in range(16):
        assert pool.context_len(seq) == 1025 + private[seq]
        assert len(pool.block_table(seq)) == 65
    # shared prefix blocks carry refcount 8
    assert all(pool.refcount[b] == 8 for b in pool.block_table(0)[:64])


def _check_invariants(pool):
    live = set()
    total_refs = 0
    for seq, table in pool.tables.items():
        assert len(table) == sizing.blocks_needed(pool.ctx[seq], pool.block_size)
        live.update(table)
        total_refs += len(table)
    assert sum(pool.refcount) == total_refs
    assert len(live) + pool.num_free() == pool.num_blocks
    assert not (live & set(pool.free_list))
    for b in range(pool.num_blocks):
        refs = sum(t.count(b) for t in pool.tables.values())
        assert pool.refcount[b] == refs


def test_random_operation_invariants():
    rng = random.Random(42)
    for trial in range(200):
        pool = BlockPool(16, rng.choice([1, 2, 4]), initial_free_order=rng.sample(range(16), 16))
        next_id = 0
        for _ in range(60):
            op = rng.random()
            live = list(pool.tables)
            try:
                if op < 0.3 or not live:
                    pool.allocate(next_id, rng.randint(0, 9))
                    next_id += 1
                elif op < 0.6:
                    pool.append_slot(rng.choice(live))
                elif op < 0.8:
                    pool.fork(rng.choice(live), next_id)
                    next_id += 1
                else:
                    pool.free(rng.choice(live))
            except PoolExhausted:
                pass
            _check_invariants(pool)


def test_planted_cow_on_full_block_is_caught():
    """A plausible mistake -- copying a shared block even when it is full -- breaks the
    beam closed form (it would add copies when the shared chain ends on a boundary)."""
    class Eager(BlockPool):
        def append_slot(self, seq):
            table = self.tables[seq]
            if table and self.refcount[table[-1]] > 1 and self.ctx[seq] % self.block_size == 0:
                old = table[-1]
                (new,) = self._take(1)
                self.refcount[old] -= 1
                table[-1] = new
            return super().append_slot(seq)
    pool = Eager(256, 16)
    pool.allocate(0, 1024)
    pool.fork(0, 1)
    pool.append_slot(1)
    assert 256 - pool.num_free() != 64 + 1   # the correct pool uses 65 blocks here
