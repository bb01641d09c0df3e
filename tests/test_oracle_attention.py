"""Pins for the oracle's paged decode attention, its split-KV merge and its cache ops.

Each pin checks the oracle against something other than itself:
* identity block table == contiguous attention by torch's scaled_dot_product_attention in
  float64 (a library special case, including its own GQA head grouping), and == a
  brute-force Python-loop implementation on tiny inputs;
* invariance under any permutation of physical blocks (the table is the only thing that
  says where a token lives);
* ctx = 1 returns the V row exactly; identical keys return the mean of V; a one-hot key
  with a large score returns that V row;
* partitions + log-sum-exp merge == single-pass softmax for every partition size;
* reshape_and_cache then gather returns the written rows; copy_blocks copies exactly.
Planted mistakes (a wrong GQA map, a dropped scale, swapped block/row indices, an
off-by-one tail) are shown to fail these pins.
"""
import math

import numpy as np
import pytest
import torch

import workloads
from oracle import attention, cache_ops, formats
from oracle.block_pool import BlockPool


def identity_layout(wl):
    """Place each sequence contiguously: block_tables[s][j] = s * T + j.  The physical
    cache is built with NumPy reshapes, independent of the oracle's gather loop."""
    n, T, B = wl.num_seqs, wl.max_blocks_per_seq, wl.block_size
    hkv, d = wl.num_kv_heads, wl.head_dim
    nan = formats.FORMATS[wl.dtype]["qnan"]
    kc = np.full((n * T, hkv, B, d), nan, dtype=np.uint16)
    vc = kc.copy()
    for s in range(n):
        a, b = wl.seq_start[s], wl.seq_start[s + 1]
        for cache, rows in ((kc, wl.keys[a:b]), (vc, wl.values[a:b])):
            pad = np.full((T * B, hkv, d), nan, dtype=np.uint16)
            pad[: b - a] = rows
            cache[s * T:(s + 1) * T] = pad.reshape(T, B, hkv, d).transpose(0, 2, 1, 3)
    tables = (np.arange(n)[:, None] * T + np.arange(T)[None, :]).astype(np.int32)
    return kc, vc, tables


def sdpa_reference(wl):
    """torch SDPA in float64, one sequence at a time, GQA by torch's own grouping."""
    outs = []
    for s in range(wl.num_seqs):
        a, b = wl.seq_start[s], wl.seq_start[s + 1]
        q = torch.from_numpy(formats.decode_bits(wl.q[s], wl.dtype))[None, :, None, :]
        k = torch.from_numpy(formats.decode_bits(wl.keys[a:b], wl.dtype)).permute(1, 0, 2)[None]
        v = torch.from_numpy(formats.decode_bits(wl.values[a:b], wl.dtype)).permute(1, 0, 2)[None]
        o = torch.nn.functional.scaled_dot_product_attention(
            q, k, v, scale=wl.scale, enable_gqa=wl.num_q_heads != wl.num_kv_heads)
        outs.append(o[0, :, 0, :].numpy())
    return np.stack(outs)


def oracle_out(wl, kc, vc, tables, seqs=None):
    out, err = attention.paged_decode(wl.q, kc, vc, tables, wl.context_lens, wl.scale,
                                      wl.block_size, wl.dtype, seqs=seqs)
    return out, err


SMALL = [
    dict(name="gqa2", context_lens=[1, 7, 16, 33, 100], dtype="fp16", num_q_heads=4,
         num_kv_heads=2, head_dim=64, block_size=16, num_blocks=64, max_context=112),
    dict(name="mha_b8", context_lens=[3, 8, 9, 40], dtype="bf16", num_q_heads=3,
         num_kv_heads=3, head_dim=32, block_size=8, num_blocks=64, max_context=48),
    dict(name="gqa4_b32", context_lens=[31, 32, 33, 65], dtype="bf16", num_q_heads=8,
         num_kv_heads=2, head_dim=16, block_size=32, num_blocks=64, max_context=96),
]


@pytest.mark.parametrize("spec", SMALL, ids=[s["name"] for s in SMALL])
def test_identity_table_equals_sdpa(spec):
    wl = workloads.custom(**spec)
    kc, vc, tables = identity_layout(wl)
    out, err = oracle_out(wl, kc, vc, tables)
    assert not err.any()
    np.testing.assert_allclose(out, sdpa_reference(wl), rtol=0, atol=1e-12)


def test_identity_table_equals_python_loops():
    wl = workloads.custom("loops", [1, 5, 18], "fp16", 4, 2, 8, 4, 16, 20, seed=3)
    kc, vc, tables = identity_layout(wl)
    out, _ = oracle_out(wl, kc, vc, tables)
    for s in range(wl.num_seqs):
        a, b = wl.seq_start[s], wl.seq_start[s + 1]
        ref = attention.contiguous_decode_loops(
            formats.decode_bits(wl.q[s], wl.dtype).tolist(),
            formats.decode_bits(wl.keys[a:b], wl.dtype).tolist(),
            formats.decode_bits(wl.values[a:b], wl.dtype).tolist(), wl.scale)
        np.testing.assert_allclose(out[s], np.array(ref), rtol=0, atol=1e-12)


def test_tiny_recipe_equals_sdpa_via_pool_placement():
    """The tiny recipe, placed through the block pool's shuffled free list and written
    with reshape_and_cache, still equals contiguous attention."""
    wl = workloads.tiny()
    kc, vc, tables = place_with_pool(wl)
    out, err = oracle_out(wl, kc, vc, tables)
    assert not err.any()
    np.testing.assert_allclose(out, sdpa_reference(wl), rtol=0, atol=1e-12)
    # 12 blocks used (1 + 1 + 3 + 7), none of them in identity order
    used = sorted({int(b) for s in range(4) for b in tables[s][: -(-int(wl.context_lens[s]) // 16)]})
    assert len(used) == 12


def place_with_pool(wl):
    """Tables from the oracle pool (shuffled free order), cache filled by the oracle's
    reshape_and_cache from the logical rows; every other slot holds NaN."""
    pool = BlockPool(wl.num_blocks, wl.block_size, wl.free_order)
    T = wl.max_blocks_per_seq
    tables = np.full((wl.num_seqs, T), -1, dtype=np.int32)
    slots = []
    for s in range(wl.num_seqs):
        pool.allocate(s, int(wl.context_lens[s]))
        t = pool.block_table(s)
        tables[s, :len(t)] = t
        slots += [pool.slot(s, i) for i in range(int(wl.context_lens[s]))]
    nan = formats.FORMATS[wl.dtype]["qnan"]
    shape = (wl.num_blocks, wl.num_kv_heads, wl.block_size, wl.head_dim)
    kc = np.full(shape, nan, dtype=np.uint16)
    vc = np.full(shape, nan, dtype=np.uint16)
    kc, vc = cache_ops.reshape_and_cache(kc, vc, wl.keys, wl.values, np.array(slots))
    return kc, vc, tables


def test_permutation_of_physical_blocks_changes_nothing():
    wl = workloads.custom("perm", [5, 16, 17, 64, 70], "bf16", 8, 2, 32, 16, 40, 80, seed=5)
    kc, vc, tables = identity_layout(wl)
    base, _ = oracle_out(wl, kc, vc, tables)
    rng = np.random.default_rng(11)
    for _ in range(3):
        nb = kc.shape[0]
        perm = rng.permutation(nb)
        kp = np.empty_like(kc)
        vp = np.empty_like(vc)
        kp[perm] = kc
        vp[perm] = vc
        tp = perm[tables].astype(np.int32)
        out, _ = oracle_out(wl, kp, vp, tp)
        np.testing.assert_array_equal(out, base)


def test_single_token_returns_v_exactly():
    wl = workloads.custom("one", [1, 1], "fp16", 4, 2, 64, 16, 8, 16, seed=7)
    kc, vc, tables = identity_layout(wl)
    out, _ = oracle_out(wl, kc, vc, tables)
    v = formats.decode_bits(wl.values, wl.dtype)           # [2, Hkv, d]
    for s in range(2):
        for h in range(4):
            np.testing.assert_array_equal(out[s, h], v[s, h // 2])
    bits, _ = attention.paged_decode_bits(wl.q, kc, vc, tables, wl.context_lens, wl.scale,
                                          wl.block_size, wl.dtype)
    np.testing.assert_array_equal(bits[:, ::2], wl.values[:, :, :])
    np.testing.assert_array_equal(bits[:, 1::2], wl.values[:, :, :])


def test_identical_keys_give_mean_of_values():
    wl = workloads.custom("same", [37], "bf16", 2, 1, 16, 8, 8, 40, seed=9)
    wl.keys[:] = wl.keys[0]
    kc, vc, tables = identity_layout(wl)
    out, _ = oracle_out(wl, kc, vc, tables)
    mean = formats.decode_bits(wl.values, wl.dtype)[:, 0, :].mean(axis=0)
    np.testing.assert_allclose(out[0, 0], mean, rtol=0, atol=1e-13)
    np.testing.assert_allclose(out[0, 1], mean, rtol=0, atol=1e-13)


def test_one_hot_key_selects_its_value_row():
    wl = workloads.custom("hot", [50], "fp16", 1, 1, 16, 16, 8, 64, scale=1.0, seed=10)
    q = np.zeros(16)
    q[3] = 8.0
    wl.q[0, 0] = formats.encode_bits(q, "fp16")
    k = np.zeros((50, 1, 16))
    k[29, 0, 3] = 8.0                                  # score 64 against 0 elsewhere
    wl.keys[:] = formats.encode_bits(k, "fp16")
    kc, vc, tables = identity_layout(wl)
    out, _ = oracle_out(wl, kc, vc, tables)
    v = formats.decode_bits(wl.values, "fp16")[29, 0]
    np.testing.assert_allclose(out[0, 0], v, rtol=0, atol=1e-20)


def test_invalid_items_give_zeros_and_flags():
    wl = workloads.custom("bad", [5, 20, 3], "fp16", 2, 1, 16, 16, 8, 32, seed=12)
    kc, vc, tables = identity_layout(wl)
    lens = wl.context_lens.copy()
    lens[0] = 0                                        # empty context
    lens[2] = 33                                       # beyond T * B
    tables = tables.copy()
    tables[1, 1] = 99                                  # block id outside the pool
    out, err = attention.paged_decode(wl.q, kc, vc, tables, lens, wl.scale, 16, "fp16")
    assert list(err) == [attention.ERR_BAD_CONTEXT, attention.ERR_BAD_BLOCK,
                         attention.ERR_BAD_CONTEXT]
    assert not out.any()


@pytest.mark.parametrize("part", [1, 8, 16, 48, 100, 1000])
def test_split_partials_merge_equals_single_pass(part):
    rng = np.random.default_rng(part)
    z = rng.standard_normal(100) * 3
    v = rng.standard_normal((100, 8))
    w = np.exp(z - z.max())
    ref = (w / w.sum()) @ v
    m, l, acc = attention.partition_partials(z, v, part)
    assert len(m) == math.ceil(100 / part)
    np.testing.assert_allclose(attention.merge_partials(m, l, acc), ref, rtol=0, atol=1e-13)


def test_split_decode_head_matches_sdpa():
    wl = workloads.custom("split", [300], "bf16", 4, 1, 32, 16, 32, 320, seed=13)
    ref = sdpa_reference(wl)
    q = formats.decode_bits(wl.q[0], "bf16")
    k = formats.decode_bits(wl.keys, "bf16")[:, 0]
    v = formats.decode_bits(wl.values, "bf16")[:, 0]
    for part in (16, 64, 256, 300):
        for h in range(4):
            o = attention.split_decode_head(q[h], k, v, wl.scale, part)
            np.testing.assert_allclose(o, ref[0, h], rtol=0, atol=1e-12)


# ----------------------------------------------------------------------------- cache ops

def test_reshape_and_cache_then_gather_returns_the_rows():
    wl = workloads.custom("w", [5, 16, 17], "bf16", 2, 2, 16, 8, 12, 24, seed=14)
    kc, vc, tables = place_with_pool(wl)
    for s in range(wl.num_seqs):
        a, b = wl.seq_start[s], wl.seq_start[s + 1]
        rows = attention.logical_rows(kc, tables[s], b - a, 8, "bf16")
        np.testing.assert_array_equal(rows, formats.decode_bits(wl.keys[a:b], "bf16"))
    # every slot not written holds NaN still
    written = sum(int(c) for c in wl.context_lens)
    assert np.isnan(formats.decode_bits(kc, "bf16")).sum() == (kc.size - written * 2 * 16)


def test_reshape_and_cache_negative_slot_skips_and_bounds():
    kc = np.zeros((2, 1, 4, 2), dtype=np.uint16)
    key = np.array([[[1, 2]], [[3, 4]]], dtype=np.uint16)
    k2, _ = cache_ops.reshape_and_cache(kc, kc, key, key, np.array([-1, 5]))
    assert k2[1, 0, 1].tolist() == [3, 4] and k2.sum() == 7
    with pytest.raises(IndexError):
        cache_ops.reshape_and_cache(kc, kc, key, key, np.array([0, 8]))
    with pytest.raises(ValueError):
        cache_ops.reshape_and_cache(kc, kc, key, key, np.array([3, 3]))


def test_copy_blocks_exact_and_rejects_alias():
    rng = np.random.default_rng(15)
    kc = rng.integers(0, 65535, size=(6, 2, 4, 3), dtype=np.uint16)
    vc = rng.integers(0, 65535, size=(6, 2, 4, 3), dtype=np.uint16)
    k2, v2 = cache_ops.copy_blocks(kc, vc, [(0, 3), (1, 4)])
    np.testing.assert_array_equal(k2[3], kc[0])
    np.testing.assert_array_equal(v2[4], vc[1])
    np.testing.assert_array_equal(k2[[0, 1, 2, 5]], kc[[0, 1, 2, 5]])
    for bad in ([(0, 3), (1, 3)], [(0, 3), (3, 4)]):
        with pytest.raises(ValueError):
            cache_ops.copy_blocks(kc, vc, bad)
    with pytest.raises(IndexError):
        cache_ops.copy_blocks(kc, vc, [(0, 6)])


# ------------------------------------------------------------------- planted mistakes

def _sdpa_pin_holds(wl):
    kc, vc, tables = identity_layout(wl)
    out, _ = oracle_out(wl, kc, vc, tables)
    return np.max(np.abs(out - sdpa_reference(wl))) < 1e-9


def test_planted_wrong_gqa_map_is_caught(monkeypatch):
    wl = workloads.custom(**SMALL[0])
    assert _sdpa_pin_holds(wl)

    def attend_modulo(q_heads, k_rows, v_rows, scale):
        hq, hkv = q_heads.shape[0], k_rows.shape[1]
        out = np.empty((hq, q_heads.shape[1]))
        for h in range(hq):
            z = scale * (k_rows[:, h % hkv, :] @ q_heads[h])
            w = np.exp(z - z.max())
            out[h] = (w / w.sum()) @ v_rows[:, h % hkv, :]
        return out
    monkeypatch.setattr(attention, "attend", attend_modulo)
    assert not _sdpa_pin_holds(wl)


def test_planted_dropped_scale_is_caught(monkeypatch):
    wl = workloads.custom(**SMALL[1])
    real = attention.attend
    monkeypatch.setattr(attention, "attend", lambda q, k, v, scale: real(q, k, v, 1.0))
    assert not _sdpa_pin_holds(wl)


def test_planted_swapped_block_and_row_is_caught(monkeypatch):
    wl = workloads.custom(**SMALL[0])

    def swapped(cache_bits, table_row, ctx, block_size, dtype):
        nb, hkv, b, d = cache_bits.shape
        out = np.empty((ctx, hkv, d))
        for t in range(ctx):
            blk = int(table_row[min(t % block_size, len(table_row) - 1)])
            out[t] = formats.decode_bits(cache_bits[blk, :, (t // block_size) % b, :], dtype)
        return out
    monkeypatch.setattr(attention, "logical_rows", swapped)
    with np.errstate(invalid="ignore"):
        assert not _sdpa_pin_holds(wl)


def test_planted_short_tail_is_caught(monkeypatch):
    wl = workloads.custom(**SMALL[0])
    real = attention.logical_rows

    def short(cache_bits, table_row, ctx, block_size, dtype):
        return real(cache_bits, table_row, max(ctx - 1, 1), block_size, dtype)
    monkeypatch.setattr(attention, "logical_rows", short)
    assert not _sdpa_pin_holds(wl)
