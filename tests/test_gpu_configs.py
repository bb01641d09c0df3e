"""The five workload recipes at full size, in the launch configuration the benchmark
times: block tables bit-exact against the oracle's placement, and every output element of
every sequence against the oracle's float64 decode of that sequence's logical rows."""
import numpy as np
import pytest
import torch

import paged_kv_cache_149_gb300 as pa
import workloads
from gpu_harness import (TOL, GpuBatch, device_error, max_err, nan_cache,
                         oracle_seq_bits, to_bits, to_device)
from oracle import attention, cache_ops, formats
from oracle.block_pool import BlockPool as OraclePool

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(libpa):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    device_error()


def oracle_tables(wl):
    pool = OraclePool(wl.num_blocks, wl.block_size, wl.free_order)
    tables = np.full((wl.num_seqs, wl.max_blocks_per_seq), -1, dtype=np.int32)
    for s in range(wl.num_seqs):
        pool.allocate(s, int(wl.context_lens[s]))
        t = pool.block_table(s)
        tables[s, :len(t)] = t
    return tables


def worst_error(wl, out_bits):
    """max |gpu - oracle| over every element of every sequence."""
    return max(max_err(out_bits[s], oracle_seq_bits(wl, s), wl.dtype) for s in range(wl.num_seqs))


@pytest.mark.parametrize("name", ["llama31_8b", "llama7b_mha", "long_b8", "long_b16", "long_b32"])
def test_recipe_full_size(name):
    wl = workloads.RECIPES[name]()
    gb = GpuBatch(wl)
    np.testing.assert_array_equal(gb.tables_np, oracle_tables(wl))
    out = to_bits(gb.decode())
    assert device_error() == 0
    assert not np.isnan(formats.decode_bits(out, wl.dtype)).any()
    worst = worst_error(wl, out)
    assert worst <= TOL[wl.dtype], f"{name}: max abs error {worst}"


def test_llama31_8b_step_writes_new_tokens_then_decodes():
    """The benchmark's step: each sequence's newest token goes through reshape_and_cache
    (64 tokens), then decode reads it."""
    wl = workloads.llama31_8b()
    n = wl.num_seqs
    # place everything, then overwrite each newest row with NaN and write it again
    gb = GpuBatch(wl)
    last = np.array([gb.pool.slots(s, int(wl.context_lens[s]) - 1, 1)[0] for s in range(n)])
    rows = wl.seq_start[1:] - 1
    nan = formats.FORMATS[wl.dtype]["qnan"]
    poison = np.full((n, wl.num_kv_heads, wl.head_dim), nan, dtype=np.uint16)
    slot_t = torch.from_numpy(last).cuda()
    pa.reshape_and_cache(to_device(poison, wl.dtype), to_device(poison, wl.dtype), gb.k_cache,
                         gb.v_cache, slot_t)
    pa.reshape_and_cache(to_device(wl.keys[rows], wl.dtype), to_device(wl.values[rows], wl.dtype),
                         gb.k_cache, gb.v_cache, slot_t)
    out = to_bits(gb.decode())
    assert device_error() == 0
    # the written rows, read back at their slots, are the newest logical rows
    kb, vb = to_bits(gb.k_cache), to_bits(gb.v_cache)
    for s in range(n):
        blk, row = divmod(int(last[s]), wl.block_size)
        np.testing.assert_array_equal(kb[blk, :, row, :], wl.keys[rows[s]])
        np.testing.assert_array_equal(vb[blk, :, row, :], wl.values[rows[s]])
    assert worst_error(wl, out) <= TOL[wl.dtype]


def test_llama31_8b_permutation_bit_identical_full_size():
    wl = workloads.llama31_8b()
    a = to_bits(GpuBatch(wl).decode())
    order = np.random.default_rng(77).permutation(wl.num_blocks).astype(np.int32)
    b = to_bits(GpuBatch(wl, free_order=order).decode())
    np.testing.assert_array_equal(a, b)


def beam_ops(pool, wl, write, copy):
    """Shared-prefix beams through a pool; `write(slots, keys, values)` and `copy(pairs)`
    apply the cache side.  Returns the final block tables and context lengths."""
    B = wl.block_size
    for p in range(wl.prompts):
        root = p * wl.beams
        pool.allocate(root, wl.shared_tokens - 1)
        slots = [pool_slot(pool, root, t, B) for t in range(wl.shared_tokens - 1)]
        s_new, cow = pool.append_slot(root)
        assert cow is None
        write(np.array(slots + [s_new], dtype=np.int64), wl.shared_keys[p], wl.shared_values[p])
        for b in range(1, wl.beams):
            pool.fork(root, root + b)
    cows, slots, keys, values = [], [], [], []
    for seq in range(wl.prompts * wl.beams):
        for i in range(int(wl.private_tokens[seq])):
            s, cow = pool.append_slot(seq)
            if cow:
                cows.append(cow)
            slots.append(s)
            keys.append(wl.private_keys[seq][i])
            values.append(wl.private_values[seq][i])
    copy(cows)
    write(np.array(slots, dtype=np.int64), np.stack(keys), np.stack(values))
    n = wl.prompts * wl.beams
    tables = np.full((n, wl.max_blocks_per_seq), -1, dtype=np.int32)
    ctx = np.zeros(n, dtype=np.int32)
    for seq in range(n):
        t = list(pool.block_table(seq))
        tables[seq, :len(t)] = t
        ctx[seq] = pool.context_len(seq)
    return tables, ctx, cows


def pool_slot(pool, seq, t, B):
    if hasattr(pool, "slot"):
        return pool.slot(seq, t)
    return int(pool.slots(seq, t, 1)[0])


def test_beam_recipe_copy_on_write():
    wl = workloads.beam()
    shape = (wl.num_blocks, wl.num_kv_heads, wl.block_size, wl.head_dim)
    # --- library side
    kc = nan_cache(*shape, wl.dtype)
    vc = nan_cache(*shape, wl.dtype)

    def gwrite(slots, k, v):
        pa.reshape_and_cache(to_device(k, wl.dtype), to_device(v, wl.dtype), kc, vc,
                             torch.from_numpy(slots).cuda())

    def gcopy(pairs):
        pa.check_block_mapping(pairs, wl.num_blocks)
        pa.copy_blocks(kc, vc, torch.tensor(pairs, dtype=torch.int32, device="cuda"))
    gtables, gctx, gcows = beam_ops(pa.BlockPool(wl.num_blocks, wl.block_size, wl.free_order),
                                    wl, gwrite, gcopy)
    assert len(gcows) == 14
    q = to_device(wl.q, wl.dtype)
    out = pa.decode(q, kc, vc, torch.from_numpy(gtables).cuda(), torch.from_numpy(gctx).cuda(),
                    wl.scale)
    assert device_error() == 0
    # --- oracle side
    nan = formats.FORMATS[wl.dtype]["qnan"]
    st = {"k": np.full(shape, nan, dtype=np.uint16), "v": np.full(shape, nan, dtype=np.uint16)}

    def owrite(slots, k, v):
        st["k"], st["v"] = cache_ops.reshape_and_cache(st["k"], st["v"], k, v, slots)

    def ocopy(pairs):
        st["k"], st["v"] = cache_ops.copy_blocks(st["k"], st["v"], pairs)
    otables, octx, ocows = beam_ops(OraclePool(wl.num_blocks, wl.block_size, wl.free_order),
                                    wl, owrite, ocopy)
    assert gcows == ocows
    np.testing.assert_array_equal(gtables, otables)
    np.testing.assert_array_equal(gctx, octx)
    np.testing.assert_array_equal(to_bits(kc), st["k"])
    np.testing.assert_array_equal(to_bits(vc), st["v"])
    ref, err = attention.paged_decode_bits(wl.q, st["k"], st["v"], otables, octx, wl.scale,
                                           wl.block_size, wl.dtype)
    assert not err.any()
    assert max_err(to_bits(out), ref, wl.dtype) <= TOL[wl.dtype]
