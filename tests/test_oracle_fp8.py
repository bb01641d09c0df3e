"""Pins for the FP8 (E4M3) KV oracle: the element format against torch.float8_e4m3fn (a
library's independent implementation of the same format), ties to even, saturation in
closed form, the quantisation error bound, and decode over FP8 blocks against the 16-bit
decode oracle on caches holding the same dequantised values; planted mistakes (the
wrong scale for V, a dropped scale) must fail."""
import math

import numpy as np
import pytest
import torch

import workloads
from oracle import attention, formats, fp8
from oracle.block_pool import BlockPool


def all_finite_codes():
    c = np.arange(256, dtype=np.uint8)
    return c[(c & 0x7F) != 0x7F]


def test_decode_every_code_matches_torch():
    c = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(c).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = fp8.decode_e4m3(c)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])
    assert fp8.decode_e4m3([0x7E])[0] == 448.0 and fp8.decode_e4m3([0x01])[0] == 2.0 ** -9
    assert fp8.decode_e4m3([0x08])[0] == 2.0 ** -6


def test_encode_matches_torch_in_range_including_every_midpoint():
    vals = np.unique(np.abs(fp8.decode_e4m3(all_finite_codes())))
    mids = (vals[:-1] + vals[1:]) / 2
    rng = np.random.default_rng(0)
    x = np.concatenate([vals, mids, -vals, -mids, rng.uniform(-448, 448, 20000),
                        rng.standard_normal(20000) * 0.01]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(fp8.encode_e4m3(x.astype(np.float64)), ref)


def test_ties_go_to_even_and_round_trip():
    # 1.0 = 0x38, 1.125 = 0x39, 1.25 = 0x3A: the midpoint 1.0625 -> 1.0, 1.1875 -> 1.25
    assert list(fp8.encode_e4m3([1.0625, 1.1875, 2.0 ** -10, 3 * 2.0 ** -10])) == [0x38, 0x3A, 0x00, 0x02]
    c = all_finite_codes()
    back = fp8.encode_e4m3(fp8.decode_e4m3(c))
    # +0 and -0 both survive; every other finite code maps to itself
    assert np.array_equal(back, c)


def test_saturation_closed_form():
    got = fp8.encode_e4m3([448.0, 449.0, 463.9, 464.0, 480.0, 1e9, math.inf, -464.0, -math.inf])
    assert list(got) == [0x7E] * 7 + [0xFE, 0xFE]
    n = fp8.encode_e4m3([math.nan, -math.nan])
    assert list(n) == [0x7F, 0xFF]


def test_quantisation_error_bound_and_exact_power_of_two_scale():
    """|decode(q(x)) * s - x| <= half a quantum of x / s (times s) inside the range, and a
    power-of-two scale only shifts exponents (q(x, 2^k) = encode(x * 2^-k))."""
    rng = np.random.default_rng(1)
    x = workloads.to_bits(rng.standard_normal(50000).astype(np.float32) * 2.0, "bf16")
    xv = formats.decode_bits(x, "bf16")
    for s in (2.0 ** -6, 0.0123, 0.5):
        codes = fp8.quantize(x, "bf16", s)
        y = fp8.decode_e4m3(codes) * float(np.float32(s))
        z = np.abs(xv / s)
        inside = z <= 448
        _, e2 = np.frexp(z)
        quantum = np.ldexp(1.0, np.maximum(e2 - 1, -6) - 3)
        # float32 division adds at most half an ulp of float32 before the E4M3 rounding
        bound = (quantum / 2 + z * 2.0 ** -24) * s
        assert np.all(np.abs(y - xv)[inside] <= bound[inside] * (1 + 1e-12))
        assert np.all(np.abs(y[~inside]) == 448 * float(np.float32(s)))
    s = 2.0 ** -6
    assert np.array_equal(fp8.quantize(x, "bf16", s), fp8.encode_e4m3(xv / s))


def place_fp8(wl, k_scale, v_scale, free_order=None):
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
    k8, v8 = np.full(shape, 0x7F, np.uint8), np.full(shape, 0x7F, np.uint8)   # NaN-filled
    k8, v8 = fp8.reshape_and_cache(k8, v8, wl.keys, wl.values, np.array(slots), k_scale,
                                   v_scale, wl.dtype)
    return k8, v8, tables


def test_decode_over_fp8_blocks_is_decode_over_the_dequantised_values():
    """Each E4M3 value times a power-of-two scale is exactly a bf16 value, so a bf16 cache
    can hold the dequantised rows; the FP8 decode must equal the 16-bit decode oracle on
    it (a different scale for K and V, so swapping them shows)."""
    wl = workloads.custom("f8b", [7, 16, 33, 100], "bf16", 4, 2, 64, 16, 64, 128, seed=1)
    ks, vs = 2.0 ** -5, 2.0 ** -3
    k8, v8, tables = place_fp8(wl, ks, vs)
    got, err = fp8.paged_decode(wl.q, k8, v8, tables, wl.context_lens, wl.scale, ks, vs,
                                wl.block_size, wl.dtype)
    assert not err.any()
    nan = formats.FORMATS["bf16"]["qnan"]
    kb = formats.encode_bits(fp8.decode_e4m3(k8) * ks, "bf16")   # NaN codes -> bf16 NaN
    vb = formats.encode_bits(fp8.decode_e4m3(v8) * vs, "bf16")
    assert np.array_equal(kb == nan, k8 == 0x7F)
    ref, err2 = attention.paged_decode(wl.q, kb, vb, tables, wl.context_lens, wl.scale,
                                       wl.block_size, "bf16")
    assert not err2.any()
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)
    # planted: V read with K's scale, or no scale at all
    bad = [attention.attend(formats.decode_bits(wl.q[s], wl.dtype),
                            fp8.logical_rows(k8, tables[s], int(wl.context_lens[s]), wl.block_size, ks),
                            fp8.logical_rows(v8, tables[s], int(wl.context_lens[s]), wl.block_size, ks),
                            wl.scale) for s in range(wl.num_seqs)]
    assert np.abs(np.stack(bad) - got).max() > 1e-3


def test_fp8_decode_against_torch_sdpa_on_an_identity_table():
    """Contiguous placement: torch's float64 attention over the dequantised rows."""
    wl = workloads.custom("f8", [5, 16, 40], "bf16", 8, 2, 64, 16, 16, 64, seed=4)
    ks, vs = 0.0123, 0.0456
    order = np.arange(wl.num_blocks, dtype=np.int32)
    k8, v8, tables = place_fp8(wl, ks, vs, free_order=order)
    got, _ = fp8.paged_decode(wl.q, k8, v8, tables, wl.context_lens, wl.scale, ks, vs,
                              wl.block_size, wl.dtype)
    g = wl.num_q_heads // wl.num_kv_heads
    for s in range(wl.num_seqs):
        a, b = wl.seq_start[s], wl.seq_start[s + 1]
        k = torch.from_numpy(fp8.decode_e4m3(fp8.quantize(wl.keys[a:b], wl.dtype, ks)) *
                             float(np.float32(ks)))
        v = torch.from_numpy(fp8.decode_e4m3(fp8.quantize(wl.values[a:b], wl.dtype, vs)) *
                             float(np.float32(vs)))
        q = torch.from_numpy(formats.decode_bits(wl.q[s], wl.dtype))[:, None, :]
        o = torch.nn.functional.scaled_dot_product_attention(
            q, k.repeat_interleave(g, dim=1).transpose(0, 1),
            v.repeat_interleave(g, dim=1).transpose(0, 1), scale=wl.scale)
        np.testing.assert_allclose(got[s], o[:, 0, :].numpy(), rtol=0, atol=1e-12)


def test_physical_permutation_changes_nothing():
    wl = workloads.tiny()
    a, _ = fp8.paged_decode(wl.q, *place_fp8(wl, 0.02, 0.03), wl.context_lens, wl.scale,
                            0.02, 0.03, wl.block_size, wl.dtype)
    order = np.random.default_rng(5).permutation(wl.num_blocks).astype(np.int32)
    b, _ = fp8.paged_decode(wl.q, *place_fp8(wl, 0.02, 0.03, order), wl.context_lens, wl.scale,
                            0.02, 0.03, wl.block_size, wl.dtype)
    np.testing.assert_array_equal(a, b)


def test_cache_write_skips_and_rejects_like_the_16_bit_one():
    rng = np.random.default_rng(2)
    key = workloads.to_bits(rng.standard_normal((3, 2, 8)).astype(np.float32), "fp16")
    k8 = np.zeros((4, 2, 4, 8), np.uint8)
    out, _ = fp8.reshape_and_cache(k8, k8, key, key, np.array([5, -1, 0]), 0.1, 0.1, "fp16")
    assert np.array_equal(out[1, :, 1], fp8.quantize(key[0], "fp16", 0.1))
    assert np.array_equal(out[0, :, 0], fp8.quantize(key[2], "fp16", 0.1))
    assert out.sum() == out[1, :, 1].astype(int).sum() + out[0, :, 0].astype(int).sum()
    with pytest.raises(ValueError):
        fp8.reshape_and_cache(k8, k8, key, key, np.array([5, 5, 0]), 0.1, 0.1, "fp16")
    with pytest.raises(IndexError):
        fp8.reshape_and_cache(k8, k8, key, key, np.array([16, 1, 0]), 0.1, 0.1, "fp16")
