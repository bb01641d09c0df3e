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
