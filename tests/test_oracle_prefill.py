"""Pins of the paged prefill oracle against things other than itself: the decode oracle
(one new token per sequence), torch's causal scaled_dot_product_attention in float64 (a
library special case: a prompt from scratch with an identity table), the tail of a full
prompt (a chunk), pure-Python loops on a tiny case, physical-block permutations, and two
planted mistakes that a pin has to catch."""
import math

import numpy as np
import pytest
import torch

import workloads
from oracle import attention, cache_ops, formats, prefill
from oracle.block_pool import BlockPool


def place(wl, free_order=None):
    """The oracle's own placement of every logical row (pool + cache write)."""
    order = wl.free_order if free_order is None else free_order
    pool = BlockPool(wl.num_blocks, wl.block_size, order)
    tables = np.full((wl.num_seqs, wl.max_blocks_per_seq), -1, dtype=np.int32)
    slots = []
    for s in range(wl.num_seqs):
        c = int(wl.context_lens[s])
        pool.allocate(s, c)
        t = pool.block_table(s)
        tables[s, :len(t)] = t
        slots += [pool.slot(s, i) for i in range(c)]
    shape = (wl.num_blocks, wl.num_kv_heads, wl.block_size, wl.head_dim)
    nan = formats.FORMATS[wl.dtype]["qnan"]
    kc = np.full(shape, nan, dtype=np.uint16)
    vc = np.full(shape, nan, dtype=np.uint16)
    kc, vc = cache_ops.reshape_and_cache(kc, vc, wl.keys, wl.values, np.array(slots, dtype=np.int64))
    return kc, vc, tables


def run(wl, free_order=None):
    kc, vc, tables = place(wl, free_order)
    return prefill.paged_prefill(wl.q, kc, vc, tables, wl.context_lens, wl.query_start,
                                 wl.scale, wl.block_size, wl.dtype)


def from_scratch(ctx, dtype="fp16", hq=4, hkv=2, d=32, seed=3):
    """Prompts from scratch: q_len = ctx for every sequence."""
    rng = np.random.default_rng(seed)
    nb = sum(-(-c // 16) for c in ctx) + 4
    return workloads._prefill("scratch", rng, ctx, ctx, dtype, hq, hkv, d, 16, nb,
                              (max(ctx) // 16 + 1) * 16, 1.0 / math.sqrt(d))


def test_one_new_token_per_sequence_is_the_decode_oracle():
    wl = workloads.tiny()
    kc, vc, tables = place(wl)
    qs = np.arange(wl.num_seqs + 1, dtype=np.int64)
    got, err = prefill.paged_prefill(wl.q, kc, vc, tables, wl.context_lens, qs, wl.scale,
                                     wl.block_size, wl.dtype)
    ref, err2 = attention.paged_decode(wl.q, kc, vc, tables, wl.context_lens, wl.scale,
                                       wl.block_size, wl.dtype)
    assert not err.any() and not err2.any()
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)


def sdpa_causal(wl, s):
    """torch float64 causal attention over sequence s's logical rows (GQA by repeating
    each kv head for its G query heads)."""
    a, b = wl.seq_start[s], wl.seq_start[s + 1]
    k = torch.from_numpy(formats.decode_bits(wl.keys[a:b], wl.dtype))        # [ctx, Hkv, d]
    v = torch.from_numpy(formats.decode_bits(wl.values[a:b], wl.dtype))
    qa, qb = wl.query_start[s], wl.query_start[s + 1]
    q = torch.from_numpy(formats.decode_bits(wl.q[qa:qb], wl.dtype))         # [ctx, Hq, d]
    g = wl.num_q_heads // wl.num_kv_heads
    k = k.repeat_interleave(g, dim=1).transpose(0, 1)
    v = v.repeat_interleave(g, dim=1).transpose(0, 1)
    o = torch.nn.functional.scaled_dot_product_attention(q.transpose(0, 1), k, v,
                                                         is_causal=True, scale=wl.scale)
    return o.transpose(0, 1).numpy()


def test_prompt_from_scratch_is_torch_causal_attention():
    wl = from_scratch([1, 7, 16, 33, 70])
    out, err = run(wl)
    assert not err.any()
    for s in range(wl.num_seqs):
        qa, qb = wl.query_start[s], wl.query_start[s + 1]
        np.testing.assert_allclose(out[qa:qb], sdpa_causal(wl, s), rtol=0, atol=1e-12)


def test_a_chunk_is_the_tail_of_the_whole_prompt():
    full = from_scratch([40, 65], seed=5)
    out_full, _ = run(full)
    # same rows, only the last `c` tokens of each sequence new
    chunks = [9, 65]
    q_rows = np.concatenate([full.q[full.query_start[s + 1] - c:full.query_start[s + 1]]
                             for s, c in enumerate(chunks)])
    qs = np.zeros(3, dtype=np.int64)
    qs[1:] = np.cumsum(chunks)
    kc, vc, tables = place(full)
    out, err = prefill.paged_prefill(q_rows, kc, vc, tables, full.context_lens, qs, full.scale,
                                     full.block_size, full.dtype)
    assert not err.any()
    for s, c in enumerate(chunks):
        tail = out_full[full.query_start[s + 1] - c:full.query_start[s + 1]]
        np.testing.assert_allclose(out[qs[s]:qs[s + 1]], tail, rtol=0, atol=1e-13)


def test_pure_python_loops_on_a_tiny_case():
    wl = workloads._prefill("loops", np.random.default_rng(8), [6], [3], "fp16", 2, 1, 4, 4, 3,
                            8, 0.5)
    out, err = run(wl)
    assert not err.any()
    k = formats.decode_bits(wl.keys, "fp16")
    v = formats.decode_bits(wl.values, "fp16")
    q = formats.decode_bits(wl.q, "fp16")
    for i in range(3):
        p = 3 + i  # positions 3, 4, 5
        for h in range(2):
            z = [0.5 * sum(float(q[i, h, j]) * float(k[t, 0, j]) for j in range(4))
                 for t in range(p + 1)]
            m = max(z)
            e = [math.exp(x - m) for x in z]
            for j in range(4):
                want = sum(e[t] * float(v[t, 0, j]) for t in range(p + 1)) / sum(e)
                assert abs(out[i, h, j] - want) < 1e-12


def test_physical_block_permutation_changes_nothing():
    wl = workloads.prefill_tiny()
    a, _ = run(wl)
    for seed in (1, 2):
        order = np.random.default_rng(seed).permutation(wl.num_blocks).astype(np.int32)
        b, _ = run(wl, free_order=order)
        np.testing.assert_array_equal(a, b)


def test_invalid_items_give_zeros_and_error_bits():
    wl = workloads.prefill_tiny()
    kc, vc, tables = place(wl)
    ctx = wl.context_lens.copy()
    ctx[0] = 3                      # q_len 5 > ctx 3
    t = tables.copy()
    t[1, 0] = wl.num_blocks         # a bad block id in sequence 1
    out, err = prefill.paged_prefill(wl.q, kc, vc, t, ctx, wl.query_start, wl.scale,
                                     wl.block_size, wl.dtype)
    assert err[0] == attention.ERR_BAD_CONTEXT and err[1] == attention.ERR_BAD_BLOCK
    assert err[2] == 0 and err[3] == 0
    assert not out[wl.query_start[0]:wl.query_start[2]].any()
    assert out[wl.query_start[2]:].any()


def _planted(wl, shift):
    """A broken copy of the oracle: the causal mask moved by `shift` positions."""
    kc, vc, tables = place(wl)
    s = 0
    ctx = int(wl.context_lens[s])
    k = attention.logical_rows(kc, tables[s], ctx, wl.block_size, wl.dtype)
    v = attention.logical_rows(vc, tables[s], ctx, wl.block_size, wl.dtype)
    q = formats.decode_bits(wl.q[:ctx], wl.dtype)
    g = wl.num_q_heads // wl.num_kv_heads
    out = np.zeros_like(q)
    for h in range(wl.num_q_heads):
        z = wl.scale * (q[:, h, :] @ k[:, h // g, :].T)
        z[np.arange(ctx)[None, :] > np.arange(ctx)[:, None] + shift] = -np.inf
        w = np.exp(z - z.max(axis=1, keepdims=True))
        out[:, h, :] = (w / w.sum(axis=1, keepdims=True)) @ v[:, h // g, :]
    return out


@pytest.mark.parametrize("shift", [10 ** 6, 1])
def test_planted_mask_mistakes_are_caught(shift):
    """No mask at all, or one position too many: the torch pin must see the difference."""
    wl = from_scratch([24], seed=9)
    bad = _planted(wl, shift)
    assert np.abs(bad - sdpa_causal(wl, 0)).max() > 1e-3
    assert np.abs(_planted(wl, 0) - sdpa_causal(wl, 0)).max() < 1e-12
