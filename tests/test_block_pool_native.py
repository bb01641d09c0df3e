"""The C++ block pool (libpa.so) against the oracle's pool, bit for bit: tables, free
list order, reference counts, slots, copy-on-write pairs and error codes."""
import random

import numpy as np
import pytest

from oracle.block_pool import BlockPool as OraclePool, PoolExhausted, UnknownSequence


def same_state(native, ref):
    assert list(native.free_list()) == ref.free_list
    assert native.num_free() == ref.num_free()
    for seq in ref.tables:
        assert list(native.block_table(seq)) == ref.block_table(seq)
        assert native.context_len(seq) == ref.context_len(seq)
    for b in range(ref.num_blocks):
        assert native.refcount(b) == ref.refcount[b]


def test_allocator_demo(libpa, golden):
    g = golden("allocator_demo.json")
    pool = libpa.BlockPool(g["num_blocks"], g["block_size"])
    ids = {"A": 0, "B": 1, "C": 2, "D": 3}
    for rid, n in g["requests"]:
        pool.allocate(ids[rid], n)
    for rid, table in g["tables_after_abc"].items():
        assert list(pool.block_table(ids[rid])) == table
    assert list(pool.free_list()) == g["free_after_abc"]
    pool.free(ids["A"])
    pool.free(ids["C"])
    assert pool.num_free() == g["free_count_after_freeing_a_and_c"]
    pool.allocate(ids["D"], g["request_d"][1])
    assert list(pool.block_table(ids["D"])) == g["table_d"]


def test_errors_map_to_the_oracle(libpa):
    pool = libpa.BlockPool(4, 16)
    pool.allocate(0, 40)
    with pytest.raises(libpa.PoolExhausted):
        pool.allocate(1, 33)
    with pytest.raises(libpa.UnknownSequence):
        pool.allocate(0, 1)
    with pytest.raises(libpa.UnknownSequence):
        pool.free(9)
    with pytest.raises(libpa.UnknownSequence):
        pool.fork(9, 10)
    with pytest.raises(libpa.PagedAttentionError):
        pool.slots(0, 30, 11)          # beyond the 40 tokens held
    assert list(pool.free_list()) == [3]


@pytest.mark.parametrize("seed", range(40))
def test_random_operations_match_oracle(libpa, seed):
    rng = random.Random(seed)
    nb = rng.choice([8, 16, 33])
    bs = rng.choice([1, 2, 4, 16])
    order = rng.sample(range(nb), nb)
    native = libpa.BlockPool(nb, bs, np.array(order))
    ref = OraclePool(nb, bs, order)
    next_id = 0
    for _ in range(120):
        live = list(ref.tables)
        op = rng.random()
        if op < 0.25 or not live:
            n = rng.randint(0, 3 * bs + 1)
            try:
                ref.allocate(next_id, n)
                want = None
            except PoolExhausted as e:
                want = e
            if want is None:
                native.allocate(next_id, n)
            else:
                with pytest.raises(libpa.PoolExhausted):
                    native.allocate(next_id, n)
            next_id += 1
        elif op < 0.65:
            seq = rng.choice(live)
            try:
                want = ref.append_slot(seq)
            except PoolExhausted:
                with pytest.raises(libpa.PoolExhausted):
                    native.append_slot(seq)
            else:
                assert native.append_slot(seq) == want
        elif op < 0.8:
            parent = rng.choice(live)
            ref.fork(parent, next_id)
            native.fork(parent, next_id)
            next_id += 1
        else:
            seq = rng.choice(live)
            ref.free(seq)
            native.free(seq)
        same_state(native, ref)
    for seq in ref.tables:
        ctx = ref.context_len(seq)
        assert list(native.slots(seq, 0, ctx)) == [ref.slot(seq, t) for t in range(ctx)]


def test_beam_script_matches_oracle(libpa):
    from test_oracle_block_pool import beam_script
    rng = random.Random(0)
    private = [rng.randint(1, 15) for _ in range(16)]
    order = list(np.random.default_rng(3).permutation(256))
    ref = OraclePool(256, 16, order)
    native = libpa.BlockPool(256, 16, np.array(order))
    ref_cows = beam_script(ref, private=private)

    class Adapter:
        def __init__(self, p):
            self.p = p

        def allocate(self, s, n):
            self.p.allocate(s, n)

        def append_slot(self, s):
            return self.p.append_slot(s)

        def fork(self, a, b):
            self.p.fork(a, b)
    nat_cows = beam_script(Adapter(native), private=private)
    assert nat_cows == ref_cows and len(nat_cows) == 14
    same_state(native, ref)


def same_tiers(native, ref):
    same_state(native, ref)
    assert list(native.cpu_free_list()) == ref.cpu_free_list
    assert native.num_free_cpu() == len(ref.cpu_free_list)
    for b in range(ref.num_cpu_blocks):
        assert native.cpu_refcount(b) == ref.cpu_refcount[b]
    for seq in ref.tables:
        assert native.is_swapped(seq) == ref.is_swapped(seq)


def test_swap_walkthrough_matches_oracle(libpa):
    native = libpa.BlockPool(8, 16, num_cpu_blocks=8)
    ref = OraclePool(8, 16, num_cpu_blocks=8)
    for p in (native, ref):
        p.allocate(0, 40)
        p.fork(0, 1)
    assert native.append_slot(1) == ref.append_slot(1)
    for group in ([1], [0]):
        assert [tuple(x) for x in native.swap_out(group)] == ref.swap_out(group)
        same_tiers(native, ref)
    assert [tuple(x) for x in native.swap_in([0, 1])] == ref.swap_in([0, 1])
    same_tiers(native, ref)


def test_swap_errors_map_to_the_oracle(libpa):
    native = libpa.BlockPool(4, 16, num_cpu_blocks=2)
    native.allocate(0, 40)
    native.allocate(1, 1)
    with pytest.raises(libpa.PoolExhausted):
        native.swap_out([0])
    with pytest.raises(libpa.WrongTier):
        native.swap_in([1])
    with pytest.raises(libpa.UnknownSequence):
        native.swap_out([7])
    with pytest.raises(libpa.PagedAttentionError):
        native.swap_out([1, 1])
    native.swap_out([1])
    with pytest.raises(libpa.WrongTier):
        native.append_slot(1)
    with pytest.raises(libpa.WrongTier):
        native.fork(1, 2)
    with pytest.raises(libpa.WrongTier):
        native.slots(1, 0, 1)
    assert native.is_swapped(1) and not native.is_swapped(0)
    assert list(native.free_list()) == [3] and native.num_free_cpu() == 1


@pytest.mark.parametrize("seed", range(30))
def test_random_operations_with_swaps_match_oracle(libpa, seed):
    from oracle.block_pool import WrongTier
    rng = random.Random(1000 + seed)
    nb, ncpu = rng.choice([8, 16, 24]), rng.choice([4, 12])
    bs = rng.choice([1, 2, 4, 16])
    order, corder = rng.sample(range(nb), nb), rng.sample(range(ncpu), ncpu)
    native = libpa.BlockPool(nb, bs, np.array(order), num_cpu_blocks=ncpu, cpu_free_order=corder)
    ref = OraclePool(nb, bs, order, num_cpu_blocks=ncpu, cpu_free_order=corder)
    errors = {PoolExhausted: libpa.PoolExhausted, WrongTier: libpa.WrongTier,
              UnknownSequence: libpa.UnknownSequence}
    next_id = 0

    def both(f_ref, f_nat, convert=lambda x: x):
        try:
            want = f_ref()
        except tuple(errors) as e:
            with pytest.raises(errors[type(e)]):
                f_nat()
            return
        assert convert(f_nat()) == want
    for _ in range(150):
        seqs = list(ref.tables)
        op = rng.random()
        if op < 0.2 or not seqs:
            n = rng.randint(0, 3 * bs + 1)
            both(lambda: ref.allocate(next_id, n), lambda: native.allocate(next_id, n))
            next_id += 1
        elif op < 0.45:
            seq = rng.choice(seqs)            # may be swapped out: WrongTier on both
            both(lambda: ref.append_slot(seq), lambda: native.append_slot(seq))
        elif op < 0.55:
            parent = rng.choice(seqs)
            both(lambda: ref.fork(parent, next_id), lambda: native.fork(parent, next_id))
            next_id += 1
        elif op < 0.85:
            group = rng.sample(seqs, rng.randint(1, min(3, len(seqs))))
            to_cpu = rng.random() < 0.5
            pairs = lambda x: [tuple(int(v) for v in p) for p in x]
            if to_cpu:
                both(lambda: ref.swap_out(group), lambda: native.swap_out(group), pairs)
            else:
                both(lambda: ref.swap_in(group), lambda: native.swap_in(group), pairs)
        else:
            seq = rng.choice(seqs)
            ref.free(seq)
            native.free(seq)
        same_tiers(native, ref)


def test_sha256_published_vectors_and_hashlib(libpa, golden):
    import hashlib
    for v in golden("sha256_vectors.json")["vectors"]:
        assert libpa.sha256(v["ascii"].encode()).hex() == v["sha256"]
    rng = np.random.default_rng(0)
    for n in list(range(0, 131)) + [1000, 4099]:   # every padding case across two blocks
        data = rng.integers(0, 256, size=n, dtype=np.uint8).tobytes()
        assert libpa.sha256(data) == hashlib.sha256(data).digest(), n


@pytest.mark.parametrize("bs", [1, 4, 16])
def test_block_hashes_match_oracle(libpa, bs):
    from oracle.block_pool import block_hashes
    rng = np.random.default_rng(bs)
    for n in [0, bs - 1, bs, 5 * bs + 3]:
        toks = rng.integers(-2 ** 31, 2 ** 31, size=n).tolist()
        for extra in (b"", b"tenant-7", bytes(range(200))):
            assert libpa.block_hashes(toks, bs, extra) == block_hashes(toks, bs, extra)


def same_cache(native, ref):
    same_tiers(native, ref)
    assert native.num_cached() == ref.num_cached()
    for b in range(ref.num_blocks):
        assert native.block_digest(b) == ref.digest_of[b]


@pytest.mark.parametrize("seed", range(30))
def test_random_operations_with_prefix_caching_match_oracle(libpa, seed):
    from oracle.block_pool import WrongTier
    rng = random.Random(5000 + seed)
    nb, bs = rng.choice([12, 24]), rng.choice([1, 2, 4])
    order = rng.sample(range(nb), nb)
    native = libpa.BlockPool(nb, bs, np.array(order), num_cpu_blocks=8)
    ref = OraclePool(nb, bs, order, num_cpu_blocks=8)
    errors = {PoolExhausted: libpa.PoolExhausted, WrongTier: libpa.WrongTier,
              UnknownSequence: libpa.UnknownSequence}

    def both(f_ref, f_nat, convert=lambda x: x):
        try:
            want = f_ref()
        except tuple(errors) as e:
            with pytest.raises(errors[type(e)]):
                f_nat()
            return
        assert convert(f_nat()) == want
    next_id = 0
    stems = [[1] * 8, [2, 1] * 4, []]
    for _ in range(150):
        seqs = list(ref.tables)
        op = rng.random()
        if op < 0.35 or not seqs:
            n = rng.randint(0, 4 * bs + 2)
            toks = (rng.choice(stems) + [rng.randint(0, 2) for _ in range(n)])[:max(n, 1)]
            extra = rng.choice([b"", b"", b"salt"])
            both(lambda: ref.allocate_prefix(next_id, toks, extra),
                 lambda: native.allocate_prefix(next_id, toks, extra))
            next_id += 1
        elif op < 0.45:
            n = rng.randint(0, 2 * bs)
            both(lambda: ref.allocate(next_id, n), lambda: native.allocate(next_id, n))
            next_id += 1
        elif op < 0.65:
            seq = rng.choice(seqs)
            both(lambda: ref.append_slot(seq), lambda: native.append_slot(seq))
        elif op < 0.72:
            parent = rng.choice(seqs)
            both(lambda: ref.fork(parent, next_id), lambda: native.fork(parent, next_id))
            next_id += 1
        elif op < 0.85:
            group = rng.sample(seqs, rng.randint(1, min(2, len(seqs))))
            pairs = lambda x: [tuple(int(v) for v in p) for p in x]
            if rng.random() < 0.5:
                both(lambda: ref.swap_out(group), lambda: native.swap_out(group), pairs)
            else:
                both(lambda: ref.swap_in(group), lambda: native.swap_in(group), pairs)
        else:
            seq = rng.choice(seqs)
            ref.free(seq)
            native.free(seq)
        same_cache(native, ref)


@pytest.mark.parametrize("seed", range(6))
def test_batch_allocation_equals_sequential_calls(libpa, seed):
    """One batched call (digests hashed in parallel) leaves the pool exactly as the same
    requests placed one by one, and returns the same cached counts, slots and tables."""
    rng = np.random.default_rng(seed)
    nb, bs = 4096, rng.choice([4, 16])
    order = rng.permutation(nb)
    system = rng.integers(0, 1000, size=64 * bs).tolist()
    batch, seq = libpa.BlockPool(nb, bs, order), libpa.BlockPool(nb, bs, order)
    ref = OraclePool(nb, bs, order.tolist())
    for rnd in range(3):
        n = int(rng.integers(1, 20))
        ids = [rnd * 100 + r for r in range(n)]
        prompts = [(system[:int(rng.integers(0, len(system)))] +
                    rng.integers(0, 1000, size=int(rng.integers(0, 5 * bs))).tolist())
                   for _ in range(n)]
        salts = [bytes([int(rng.integers(0, 2))]) * int(rng.integers(0, 3)) for _ in range(n)]
        ts = np.zeros(n + 1, dtype=np.int64)
        np.cumsum([len(p) for p in prompts], out=ts[1:])
        es = np.zeros(n + 1, dtype=np.int64)
        np.cumsum([len(x) for x in salts], out=es[1:])
        cached, slots, tables = batch.allocate_prefix_batch(
            ids, np.concatenate([np.asarray(p, np.int32) for p in prompts] + [np.zeros(0, np.int32)]),
            ts, b"".join(salts), es, table_width=80)
        want_slots = []
        for r, (i, p, x) in enumerate(zip(ids, prompts, salts)):
            c = seq.allocate_prefix(i, p, x)
            assert c == cached[r] == ref.allocate_prefix(i, p, x)
            want_slots.append(seq.slots(i, c, len(p) - c))
            t = seq.block_table(i)
            assert list(tables[r][:len(t)]) == list(t) and not tables[r][len(t):].any()
        np.testing.assert_array_equal(slots, np.concatenate(want_slots))
        same_cache(batch, ref)
        drop = ids[::2]
        batch.free_batch(drop)
        for i in drop:
            seq.free(i)
            ref.free(i)
        same_cache(batch, ref)


def test_hashed_batch_equals_token_batch(libpa):
    """Placing from digests computed earlier gives the pool, hits, slots and tables that
    placing from the tokens does."""
    rng = np.random.default_rng(11)
    nb, bs = 2048, 16
    order = rng.permutation(nb)
    a, b = libpa.BlockPool(nb, bs, order), libpa.BlockPool(nb, bs, order)
    system = rng.integers(0, 1000, size=40 * bs).tolist()
    for rnd in range(4):
        n = int(rng.integers(1, 12))
        ids = [rnd * 100 + r for r in range(n)]
        prompts = [system[:int(rng.integers(0, len(system)))] +
                   rng.integers(0, 1000, size=int(rng.integers(0, 4 * bs))).tolist() for _ in range(n)]
        ts = np.zeros(n + 1, dtype=np.int64)
        np.cumsum([len(p) for p in prompts], out=ts[1:])
        toks = np.concatenate([np.asarray(p, np.int32) for p in prompts] + [np.zeros(0, np.int32)])
        want = a.allocate_prefix_batch(ids, toks, ts, table_width=48)
        digests = b"".join(d for p in prompts for d in libpa.block_hashes(p, bs))
        got = b.allocate_hashed_batch(ids, [len(p) for p in prompts], digests, 48)
        for x, y in zip(want, got):
            np.testing.assert_array_equal(x, y)
        assert list(a.free_list()) == list(b.free_list()) and a.num_cached() == b.num_cached()
        a.free_batch(ids[::3])
        b.free_batch(ids[::3])


@pytest.mark.parametrize("seed", range(4))
def test_cache_churn_keeps_every_lookup_right(libpa, seed):
    """A full cache under steady churn: one-token blocks, prompts drawn from a small set of
    token runs so that hits, partial hits and misses all happen, and most allocations evict
    the oldest cached block.  Every answer (tokens found cached, tables) and the digest of
    every block match the oracle's pool, whose lookups are a plain dictionary."""
    rng = random.Random(9000 + seed)
    nb = rng.choice([61, 64, 100])
    order = rng.sample(range(nb), nb)
    native = libpa.BlockPool(nb, 1, np.array(order))
    ref = OraclePool(nb, 1, order)
    live = []
    for i in range(1500):
        toks = [rng.randint(0, 5) for _ in range(rng.randint(1, 4))]
        if ref.num_free() < 4 or (live and rng.random() < 0.45):
            seq = live.pop(rng.randrange(len(live)))
            ref.free(seq)
            native.free(seq)
            continue
        assert native.allocate_prefix(i, toks) == ref.allocate_prefix(i, toks)
        assert list(native.block_table(i)) == ref.block_table(i)
        live.append(i)
        if i % 50 == 0:
            same_cache(native, ref)
    same_cache(native, ref)
    assert ref.num_cached() > nb // 2


def test_batch_calls_refuse_buffers_too_small(libpa):
    """The library writes into caller arrays and reads caller spans by offsets: the binding
    refuses arrays too small, of the wrong type, or offsets past their data, before the
    call, and the pool is left as it was."""
    bs = 4
    pool = libpa.BlockPool(32, bs, np.arange(32))
    toks = np.arange(20, dtype=np.int32)
    ts = np.array([0, 9, 20], dtype=np.int64)
    digests = b"".join(d for a, b in ((0, 9), (9, 20)) for d in libpa.block_hashes(toks[a:b], bs))
    good = (np.zeros(2, np.int32), np.zeros(20, np.int64), np.zeros((2, 3), np.int32))
    bad_outs = [
        (np.zeros(1, np.int32), good[1], good[2]),
        (good[0], np.zeros(19, np.int64), good[2]),
        (good[0], good[1], np.zeros((2, 2), np.int32)),
        (good[0], np.zeros(20, np.int32), good[2]),
        (good[0], np.zeros(40, np.int64)[::2], good[2]),
    ]
    for out in bad_outs:
        with pytest.raises(ValueError):
            pool.allocate_prefix_batch([0, 1], toks, ts, table_width=3, out=out)
        with pytest.raises(ValueError):
            pool.allocate_hashed_batch([0, 1], [9, 11], digests, 3, out=out)
    with pytest.raises(ValueError):
        pool.allocate_prefix_batch([0, 1], toks, np.array([0, 9, 21]), table_width=3)
    with pytest.raises(ValueError):
        pool.allocate_prefix_batch([0, 1], toks, ts, extras=b"ab", extra_start=[0, 1, 3],
                                   table_width=3)
    with pytest.raises(ValueError):
        pool.allocate_hashed_batch([0, 1], [9, 11], digests[:-1], 3)
    assert pool.num_free() == 32 and pool.num_cached() == 0
    cached, slots, tables = pool.allocate_hashed_batch([0, 1], [9, 11], digests, 3, out=good)
    assert list(cached) == [0, 0] and len(slots) == 20 and tables.shape == (2, 3)


def test_batch_placement_rejects_bad_offsets_in_the_library(libpa):
    """The C entry point itself (no binding checks in front) refuses a negative first offset
    or a decreasing one, for tokens and extra bytes, and changes nothing."""
    import ctypes
    lib = libpa.lib()
    pool = libpa.BlockPool(16, 4, np.arange(16))
    ids = np.array([0, 1], dtype=np.int64)
    toks = np.arange(12, dtype=np.int32)
    extras = np.frombuffer(b"abcdef", dtype=np.uint8).copy()
    cached = np.zeros(2, dtype=np.int32)
    done = ctypes.c_int(-1)

    def call(ts, es=None):
        ts = np.asarray(ts, dtype=np.int64)
        es = None if es is None else np.asarray(es, dtype=np.int64)
        return lib.pa_pool_allocate_prefix_batch(
            pool._h, 2, ids.ctypes.data, toks.ctypes.data, ts.ctypes.data,
            None if es is None else extras.ctypes.data, None if es is None else es.ctypes.data,
            cached.ctypes.data, None, None, 0, ctypes.byref(done))
    for ts, es in (([-4, 4, 12], None), ([0, 8, 4], None), ([0, 4, 12], [-1, 2, 6]),
                   ([0, 4, 12], [0, 4, 2])):
        assert call(ts, es) == libpa.PA_ERR_ARG
        assert done.value == 0 and pool.num_free() == 16
    assert call([0, 4, 12], [0, 2, 6]) == 0 and done.value == 2 and pool.num_free() == 13


def test_table_width_is_the_widest_request(libpa):
    """pa_pool_table_width: the most blocks one request of the batch takes, ceil(len / B),
    checked against the pages' N = ceil(S / B) on the printed examples and brute force."""
    import ctypes
    import numpy as np
    for B, lens in ((16, [1000, 19, 0, 256]), (8, [1000]), (32, [1000, 31, 33]), (16, [])):
        pool = libpa.BlockPool(64, B)
        ts = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
        want = max([-(-x // B) for x in lens], default=0)
        got = libpa.lib().pa_pool_table_width(pool._h, len(lens), ts.ctypes.data)
        assert got == want, (B, lens, got)
    # 1000 tokens: 63 blocks at B = 16 (the pages' worked example)
    pool = libpa.BlockPool(64, 16)
    ts = np.array([0, 1000], np.int64)
    assert libpa.lib().pa_pool_table_width(pool._h, 1, ts.ctypes.data) == 63
    bad = np.array([0, 10, 5], np.int64)     # a decreasing offset
    assert libpa.lib().pa_pool_table_width(pool._h, 2, bad.ctypes.data) == libpa.PA_ERR_ARG
    neg = np.array([-1, 10], np.int64)
    assert libpa.lib().pa_pool_table_width(pool._h, 1, neg.ctypes.data) == libpa.PA_ERR_ARG
    assert libpa.lib().pa_pool_table_width(None, 1, ts.ctypes.data) == libpa.PA_ERR_ARG
