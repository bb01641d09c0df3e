"""Pins for automatic prefix caching in the oracle pool (chenyuan1125
"vllm-pagedattention", sections 一块内存，如何安全地属于多条序列 and 分页不是免费午餐):
the hash chain's dependence structure, salt isolation, hand-worked walk-throughs of
lookup / reuse / eviction, per-pool conservation under random operations, and the
property that makes reuse correct -- every row a request reads through a cache hit
equals the row it would have computed itself -- with planted mistakes it must catch."""
import random

import pytest

from oracle.block_pool import BlockPool, PoolExhausted, block_hashes
from test_oracle_swap import check_tiers


def test_sha256_of_the_published_vectors(golden):
    import hashlib
    for v in golden("sha256_vectors.json")["vectors"]:
        assert hashlib.sha256(v["ascii"].encode()).hexdigest() == v["sha256"]


def test_chain_dependence():
    """Block i's digest depends on every token up to the end of block i and on nothing
    after it; a partial tail block has no digest."""
    B = 4
    base = list(range(100, 118))                  # 4 full blocks + 2 tokens
    d0 = block_hashes(base, B)
    assert len(d0) == 4 and len(set(d0)) == 4
    for pos in range(18):
        t = list(base)
        t[pos] += 1
        d = block_hashes(t, B)
        blk = pos // B
        assert d[:blk] == d0[:blk]                 # earlier blocks unchanged
        assert all(a != b for a, b in zip(d[blk:], d0[blk:]))   # this one and all later
    # the same block of tokens after a different prefix is a different block
    a = block_hashes([1, 2, 3, 4, 9, 9, 9, 9], B)
    b = block_hashes([5, 6, 7, 8, 9, 9, 9, 9], B)
    assert a[1] != b[1]
    # block size is part of the identity
    assert block_hashes(list(range(8)), 4)[1] != block_hashes(list(range(8)), 8)[0]


def test_salt_separates_tenants():
    pool = BlockPool(16, 4)
    prompt = list(range(12))
    assert pool.allocate_prefix("t1-a", prompt, b"tenant-1") == 0
    assert pool.allocate_prefix("t2-a", prompt, b"tenant-2") == 0     # no cross-tenant hit
    assert pool.allocate_prefix("t1-b", prompt, b"tenant-1") == 12
    assert pool.block_table("t1-b") == pool.block_table("t1-a")
    assert not set(pool.block_table("t2-a")) & set(pool.block_table("t1-a"))


def test_walkthrough_share_miss_evict_revive():
    # 8 blocks of 4 tokens, free list 0..7
    pool = BlockPool(8, 4)
    sys_prompt = [7] * 8                           # 2 full blocks
    assert pool.allocate_prefix("A", sys_prompt + [1, 2, 3]) == 0      # 0, 1, 2
    assert pool.block_table("A") == [0, 1, 2] and pool.num_cached() == 2
    assert pool.allocate_prefix("B", sys_prompt + [4, 5, 6, 7, 8]) == 8  # hits 0, 1; new 3, 4
    assert pool.block_table("B") == [0, 1, 3, 4]
    assert [pool.refcount[b] for b in range(5)] == [2, 2, 1, 1, 1]
    assert pool.num_cached() == 3                  # + B's third block [4, 5, 6, 7]
    # the lookup stops at the first miss: same first block, different second
    assert pool.allocate_prefix("C", [7] * 4 + [0] * 4) == 4          # hit 0; new 5
    assert pool.block_table("C") == [0, 5]
    pool.free("A")
    pool.free("B")
    pool.free("C")
    # every block at count zero joins the tail in free order, cached ones included:
    # A frees 2; B frees 1, 3, 4; C frees 0, 5
    assert pool.free_list == [6, 7, 2, 1, 3, 4, 0, 5]
    assert pool.num_cached() == 4                  # 0, 1, 3, 5
    # a hit revives a cached free block from the middle of the list
    assert pool.allocate_prefix("D", sys_prompt) == 8
    assert pool.block_table("D") == [0, 1] and pool.free_list == [6, 7, 2, 3, 4, 5]
    # plain allocation takes from the head and evicts what it takes: 6, 7, 2, 3
    pool.allocate("E", 16)
    assert pool.block_table("E") == [6, 7, 2, 3] and pool.num_cached() == 3   # 3 evicted
    assert pool.allocate_prefix("F", sys_prompt + [4, 5, 6, 7]) == 8        # block 3 gone
    assert pool.block_table("F") == [0, 1, 4]


def test_exhaustion_changes_nothing():
    pool = BlockPool(4, 4)
    pool.allocate_prefix("A", list(range(8)))     # 0, 1 cached
    pool.free("A")
    pool.allocate("X", 4)                          # takes 2
    before = (list(pool.free_list), dict(pool.cached), list(pool.refcount))
    with pytest.raises(PoolExhausted):
        pool.allocate_prefix("B", list(range(8)) + [0] * 9)   # 2 hits + 3 new > 1 free
    assert (pool.free_list, pool.cached, pool.refcount) == before


def row_value(prefix):
    """The K/V 'row' a model would compute at the last position of `prefix`: any function
    of the whole prefix (two 16-bit rolling hashes)."""
    a = b = 1
    for t in prefix:
        a = (a * 31 + t + 1) % 65521
        b = (b * 131 + 7 * t + 3) % 65519
    return (a, b)


class Model:
    """A pool with its cache rows: a request writes rows only for positions it does not
    find cached; decode appends write their own rows."""

    def __init__(self, pool):
        self.pool = pool
        self.rows = {}                             # slot -> row
        self.tokens = {}                           # seq -> token list

    def prefill(self, seq, tokens, extra=b""):
        cached = self.pool.allocate_prefix(seq, tokens, extra)
        for p in range(cached, len(tokens)):
            self.rows[self.pool.slot(seq, p)] = row_value(tokens[:p + 1])
        self.tokens[seq] = list(tokens)
        return cached

    def append(self, seq, token):
        slot, cow = self.pool.append_slot(seq)
        if cow is not None:
            s, d = cow
            B = self.pool.block_size
            for r in range(B):
                if s * B + r in self.rows:
                    self.rows[d * B + r] = self.rows[s * B + r]
        self.tokens[seq].append(token)
        self.rows[slot] = row_value(self.tokens[seq])

    def check(self):
        for seq, toks in self.tokens.items():
            for p in range(len(toks)):
                assert self.rows.get(self.pool.slot(seq, p)) == row_value(toks[:p + 1]), (seq, p)


def random_prefix_ops(pool, rng, steps, model):
    vocab = [0, 1, 2]                               # few tokens: many shared prefixes
    for _ in range(steps):
        live = list(pool.tables)
        op = rng.random()
        try:
            if op < 0.4 or not live:
                seq = max(live + [0]) + 1
                n = rng.randint(0, 4 * pool.block_size + 2)
                stem = rng.choice([[1] * 8, [2, 1] * 4, []])
                toks = (stem + [rng.choice(vocab) for _ in range(n)])[:max(n, 1)]
                model.prefill(seq, toks, rng.choice([b"", b"", b"s"]))
            elif op < 0.7:
                model.append(rng.choice(live), rng.choice(vocab))
            elif op < 0.8:
                parent = rng.choice(live)
                child = max(live) + 1
                pool.fork(parent, child)
                model.tokens[child] = list(model.tokens[parent])
            else:
                seq = rng.choice(live)
                pool.free(seq)
                del model.tokens[seq]
        except PoolExhausted:
            pass
        check_tiers(pool)
        for dg, b in pool.cached.items():
            assert pool.digest_of[b] == dg
        model.check()


def test_random_operations_reuse_is_always_correct():
    rng = random.Random(5)
    for _ in range(120):
        pool = BlockPool(rng.choice([12, 24]), rng.choice([2, 4]))
        random_prefix_ops(pool, rng, 60, Model(pool))


def test_planted_mistakes_are_caught():
    """(1) Hashing each block without its parent lets a block be reused after a different
    prefix; (2) forgetting to evict a digest when its block is taken for other use leaves
    a stale mapping.  Both serve wrong rows, which the reuse check sees."""
    import oracle.block_pool as bp

    def unchained(tokens, block_size, extra=b""):
        import hashlib
        return [hashlib.sha256(bytes(str(tokens[i * block_size:(i + 1) * block_size]), "ascii")
                               + bytes(extra)).digest()
                for i in range(len(tokens) // block_size)]

    class NoEvict(BlockPool):
        def _evict(self, b):
            pass

    for plant in ("unchained", "no_evict"):
        caught = False
        rng = random.Random(9)
        saved = bp.block_hashes
        try:
            if plant == "unchained":
                bp.block_hashes = unchained
            for _ in range(60):
                pool = (NoEvict if plant == "no_evict" else BlockPool)(12, 2)
                try:
                    random_prefix_ops(pool, rng, 60, Model(pool))
                except AssertionError:
                    caught = True
                    break
        finally:
            bp.block_hashes = saved
        assert caught, plant
