"""Pins for the INT4 KV oracle: a hand-worked row (codes, ties to even, nibble order), the
all-zero row, the quantisation error bound, exactness under power-of-two scaling, decode
over INT4 blocks against torch's float64 attention on the dequantised rows, invariance
under physical permutation; planted mistakes (K and V scales swapped, nibbles swapped)
must fail."""
import numpy as np
import pytest
import torch

import workloads
from oracle import formats, int4
from oracle.block_pool import BlockPool


def bits(x, dtype="fp16"):
    return workloads.to_bits(np.asarray(x, dtype=np.float32), dtype)


def test_hand_worked_row():
    # max |x| = 7, so s = 1 and the codes are x rounded half to even: 3.5 -> 4,
    # -3.5 -> -4, 2.5 -> 2, 0.5 -> 0, 1.5 -> 2.  Nibbles u = c + 8 = 15, 1, 12, 4, 10, 8,
    # 10, 8; element 2i is the low nibble of byte i.
    packed, s = int4.quantize_rows(bits([7, -7, 3.5, -3.5, 2.5, 0.5, 1.5, 0]), "fp16")
    assert s == np.float32(1.0)
    assert list(packed) == [0x1F, 0x4C, 0x8A, 0x8A]
    assert list(int4.unpack_codes(packed)) == [7, -7, 4, -4, 2, 0, 2, 0]


def test_zero_row_and_scale_division():
    packed, s = int4.quantize_rows(bits(np.zeros(16), "bf16"), "bf16")
    assert s == 0.0 and np.all(packed == 0x88)
    # s is max|x| / 7 rounded once to float32: for max 1.0 that is float32(1/7)
    _, s = int4.quantize_rows(bits([1.0, -0.5, 0.25, 0.0], "bf16"), "bf16")
    assert s == np.float32(1.0) / np.float32(7.0) and s != np.float64(1.0) / 7.0


def test_error_bound_and_extremes():
    """|c s - x| <= s/2 (plus float32 rounding of x/s), and the largest |x| gets |c| = 7."""
    rng = np.random.default_rng(0)
    for dtype in ("fp16", "bf16"):
        x = bits(rng.standard_normal((500, 4, 128)) * rng.uniform(0.01, 30, (500, 4, 1)), dtype)
        packed, s = int4.quantize_rows(x, dtype)
        xv = formats.decode_bits(x, dtype)
        deq = int4.dequantize(packed, s)
        s64 = s.astype(np.float64)[..., None]
        assert np.all(np.abs(deq - xv) <= s64 * (0.5 + 2.0 ** -20))
        c = int4.unpack_codes(packed)
        imax = np.argmax(np.abs(xv), axis=-1)
        assert np.all(np.abs(np.take_along_axis(c, imax[..., None], -1)) == 7)
        assert c.min() >= -7 and c.max() <= 7


def test_power_of_two_scaling_is_exact():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((64, 128)).astype(np.float32)
    p1, s1 = int4.quantize_rows(bits(x, "bf16"), "bf16")
    p2, s2 = int4.quantize_rows(bits(x * 8.0, "bf16"), "bf16")
    assert np.array_equal(p1, p2) and np.array_equal(s2, s1 * np.float32(8.0))


def place_int4(wl, free_order=None):
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
    nb, hkv, b, d = wl.num_blocks, wl.num_kv_heads, wl.block_size, wl.head_dim
    kc = np.zeros((nb, hkv, b, d // 2), np.uint8)
    ks = np.full((nb, hkv, b), np.nan, np.float32)   # never read outside the contexts
    kc, vc, ks, vs = int4.reshape_and_cache(kc, kc.copy(), ks, ks.copy(), wl.keys, wl.values,
                                            np.array(slots), wl.dtype)
    return kc, vc, ks, vs, tables


def test_decode_against_torch_sdpa_on_an_identity_table():
    wl = workloads.custom("i4", [5, 16, 40], "bf16", 8, 2, 64, 16, 16, 64, seed=4)
    kc, vc, ks, vs, tables = place_int4(wl, free_order=np.arange(16, dtype=np.int32))
    got, err = int4.paged_decode(wl.q, kc, vc, ks, vs, tables, wl.context_lens, wl.scale,
                                 wl.block_size, wl.dtype)
    assert not err.any()
    g = wl.num_q_heads // wl.num_kv_heads
    for s in range(wl.num_seqs):
        a, b = wl.seq_start[s], wl.seq_start[s + 1]
        k = torch.from_numpy(int4.dequantize(*int4.quantize_rows(wl.keys[a:b], wl.dtype)))
        v = torch.from_numpy(int4.dequantize(*int4.quantize_rows(wl.values[a:b], wl.dtype)))
        q = torch.from_numpy(formats.decode_bits(wl.q[s], wl.dtype))[:, None, :]
        o = torch.nn.functional.scaled_dot_product_attention(
            q, k.repeat_interleave(g, dim=1).transpose(0, 1),
            v.repeat_interleave(g, dim=1).transpose(0, 1), scale=wl.scale)
        np.testing.assert_allclose(got[s], o[:, 0, :].numpy(), rtol=0, atol=1e-12)
    # planted: K and V scales swapped, or the two nibbles of every byte swapped
    bad, _ = int4.paged_decode(wl.q, kc, vc, vs, ks, tables, wl.context_lens, wl.scale,
                               wl.block_size, wl.dtype)
    assert np.abs(bad - got).max() > 1e-3
    swap = lambda p: ((p >> 4) | (p << 4)).astype(np.uint8)
    bad, _ = int4.paged_decode(wl.q, swap(kc), swap(vc), ks, vs, tables, wl.context_lens,
                               wl.scale, wl.block_size, wl.dtype)
    assert np.abs(bad - got).max() > 1e-3


def test_physical_permutation_changes_nothing():
    wl = workloads.tiny()
    a, _ = int4.paged_decode(wl.q, *place_int4(wl), wl.context_lens, wl.scale, wl.block_size,
                             wl.dtype)
    order = np.random.default_rng(5).permutation(wl.num_blocks).astype(np.int32)
    b, _ = int4.paged_decode(wl.q, *place_int4(wl, order), wl.context_lens, wl.scale,
                             wl.block_size, wl.dtype)
    np.testing.assert_array_equal(a, b)


def test_one_token_context_returns_its_dequantised_value_row():
    wl = workloads.custom("i4one", [1, 1], "fp16", 4, 2, 64, 16, 8, 16, seed=2)
    kc, vc, ks, vs, tables = place_int4(wl)
    got, _ = int4.paged_decode(wl.q, kc, vc, ks, vs, tables, wl.context_lens, wl.scale,
                               wl.block_size, wl.dtype)
    for s in range(2):
        v = int4.dequantize(*int4.quantize_rows(wl.values[wl.seq_start[s]], wl.dtype))
        np.testing.assert_array_equal(got[s], np.repeat(v, 2, axis=0))


def test_cache_write_skips_and_rejects():
    rng = np.random.default_rng(2)
    key = bits(rng.standard_normal((3, 2, 8)), "fp16")
    kc = np.zeros((4, 2, 4, 4), np.uint8)
    ks = np.zeros((4, 2, 4), np.float32)
    out = int4.reshape_and_cache(kc, kc, ks, ks, key, key, np.array([5, -1, 0]), "fp16")
    p, s = int4.quantize_rows(key[0], "fp16")
    assert np.array_equal(out[0][1, :, 1], p) and np.array_equal(out[2][1, :, 1], s)
    assert out[0].astype(int).sum() == (out[0][1, :, 1].astype(int).sum() +
                                        out[0][0, :, 0].astype(int).sum())
    with pytest.raises(ValueError):
        int4.reshape_and_cache(kc, kc, ks, ks, key, key, np.array([5, 5, 0]), "fp16")
    with pytest.raises(IndexError):
        int4.reshape_and_cache(kc, kc, ks, ks, key, key, np.array([16, 1, 0]), "fp16")
