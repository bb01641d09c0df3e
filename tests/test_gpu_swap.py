"""GPU parity of swap-out / swap-in: pa_swap_blocks between a device pool and a pinned
CPU pool (and between two device pools) is bit-exact against the oracle's block copy;
bad pairs are skipped and flagged; a batch preempted, overwritten and brought back by
the C++ pool decodes bit-identically to the batch before the swap, and within the
decode tolerance of the oracle."""
import numpy as np
import pytest
import torch

import paged_kv_cache_149_gb300 as pa
import workloads
from gpu_harness import TOL, GpuBatch, device_error, max_err, oracle_place, to_bits, to_device
from oracle import attention, cache_ops

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(libpa):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    device_error()


def pools(rng, nb, hkv, bs, d):
    return (rng.integers(0, 65535, size=(nb, hkv, bs, d), dtype=np.uint16),
            rng.integers(0, 65535, size=(nb, hkv, bs, d), dtype=np.uint16))


def pinned(bits, dtype):
    return to_device(bits, dtype, "cpu").pin_memory()


def pairs_for(rng, nsrc, ndst, n):
    src = rng.integers(0, nsrc, size=n)
    dst = rng.permutation(ndst)[:n]
    return np.stack([src, dst], axis=1).astype(np.int32)


@pytest.mark.parametrize("dtype,hkv,d,bs", [("bf16", 8, 128, 16), ("fp16", 2, 64, 8),
                                             ("bf16", 1, 64, 32), ("fp16", 32, 128, 16)])
@pytest.mark.parametrize("mapping_on", ["cuda", "pinned"])
def test_swap_out_and_in_bit_exact(dtype, hkv, d, bs, mapping_on):
    rng = np.random.default_rng(hkv * 7 + d + bs)
    nb, ncpu = 48, 40
    dk, dv = pools(rng, nb, hkv, bs, d)
    ck, cv = pools(rng, ncpu, hkv, bs, d)
    gk, gv = to_device(dk, dtype), to_device(dv, dtype)
    hk, hv = pinned(ck, dtype), pinned(cv, dtype)

    def mapping(p):
        t = torch.from_numpy(p)
        return t.cuda() if mapping_on == "cuda" else t.pin_memory()
    out_pairs = pairs_for(rng, nb, ncpu, 23)
    pa.swap_blocks(gk, gv, hk, hv, mapping(out_pairs))
    torch.cuda.synchronize()
    want_ck, want_cv = cache_ops.swap_blocks(dk, dv, ck, cv, out_pairs)
    np.testing.assert_array_equal(to_bits(hk), want_ck)
    np.testing.assert_array_equal(to_bits(hv), want_cv)
    in_pairs = pairs_for(rng, ncpu, nb, 31)
    pa.swap_blocks(hk, hv, gk, gv, mapping(in_pairs))
    torch.cuda.synchronize()
    want_dk, want_dv = cache_ops.swap_blocks(want_ck, want_cv, dk, dv, in_pairs)
    np.testing.assert_array_equal(to_bits(gk), want_dk)
    np.testing.assert_array_equal(to_bits(gv), want_dv)
    assert device_error() == 0


def test_device_to_device_pools_bit_exact():
    rng = np.random.default_rng(3)
    ak, av = pools(rng, 30, 8, 16, 128)
    bk, bv = pools(rng, 20, 8, 16, 128)
    gak, gav, gbk, gbv = (to_device(x, "bf16") for x in (ak, av, bk, bv))
    p = pairs_for(rng, 30, 20, 20)
    pa.swap_blocks(gak, gav, gbk, gbv, torch.from_numpy(p).cuda())
    want_k, want_v = cache_ops.swap_blocks(ak, av, bk, bv, p)
    np.testing.assert_array_equal(to_bits(gbk), want_k)
    np.testing.assert_array_equal(to_bits(gbv), want_v)
    assert device_error() == 0


def test_bad_pairs_are_skipped_and_flagged():
    rng = np.random.default_rng(4)
    dk, dv = pools(rng, 8, 2, 16, 64)
    ck, cv = pools(rng, 4, 2, 16, 64)
    gk, gv = to_device(dk, "fp16"), to_device(dv, "fp16")
    hk, hv = pinned(ck, "fp16"), pinned(cv, "fp16")
    p = np.array([(0, 1), (8, 2), (3, 4), (5, -1), (7, 3)], dtype=np.int32)
    pa.swap_blocks(gk, gv, hk, hv, torch.from_numpy(p).cuda())
    assert device_error() == pa.DEVERR_BAD_PAIR
    want_k, want_v = cache_ops.swap_blocks(dk, dv, ck, cv, p[[0, 4]])
    np.testing.assert_array_equal(to_bits(hk), want_k)
    np.testing.assert_array_equal(to_bits(hv), want_v)


def test_pageable_host_memory_is_refused():
    """The library resolves every pointer; ordinary (pageable) host memory has no device
    address and is refused before anything is launched."""
    k = np.zeros((4, 2, 16, 64), dtype=np.uint16)
    g = torch.zeros((4, 2, 16, 64), dtype=torch.float16, device="cuda")
    m = torch.zeros((1, 2), dtype=torch.int32, device="cuda")
    st = pa.lib().pa_swap_blocks(g.data_ptr(), g.data_ptr(), k.ctypes.data, k.ctypes.data,
                                 m.data_ptr(), 1, 4, 4, 2, 64, 16, pa.PA_FP16,
                                 torch.cuda.current_stream().cuda_stream)
    assert st == pa.PA_ERR_ARG


@pytest.mark.parametrize("recipe", ["tiny", "llama"])
def test_preempt_overwrite_resume_decodes_the_same(recipe):
    """Swap out half the batch, let other requests take (and overwrite) the freed device
    blocks, swap back in: the decode equals the decode before the swap bit for bit (same
    logical rows; the kernel's result does not depend on where blocks sit) and stays
    within tolerance of the oracle."""
    if recipe == "tiny":
        wl = workloads.tiny()
    else:
        wl = workloads.custom("swap", list(np.random.default_rng(1).integers(128, 2049, 24)),
                              "bf16", 32, 8, 128, 16, 4096, 2048, seed=6)
    gb = GpuBatch(wl)
    before = to_bits(gb.decode())
    # the same placement again, in a pool with a CPU side
    pool = pa.BlockPool(wl.num_blocks, wl.block_size, wl.free_order, num_cpu_blocks=wl.num_blocks)
    for s in range(wl.num_seqs):
        pool.allocate(s, int(wl.context_lens[s]))
        assert list(pool.block_table(s)) == list(gb.tables_np[s][:len(pool.block_table(s))])
    hk = torch.empty(gb.k_cache.shape, dtype=gb.k_cache.dtype).pin_memory()
    hv = torch.empty_like(hk).pin_memory()
    group = list(range(0, wl.num_seqs, 2))
    out_pairs = pool.swap_out(group)
    pa.swap_blocks(gb.k_cache, gb.v_cache, hk, hv, torch.from_numpy(out_pairs).cuda())
    # another request takes every free device block (the freed ones among them), fills
    # them and ends, so the swap-in lands in blocks that hold its rows
    intruder = 10_000
    n_int = pool.num_free() * wl.block_size
    pool.allocate(intruder, n_int)
    slots = torch.from_numpy(pool.slots(intruder, 0, n_int)).cuda()
    junk = torch.randn((n_int, wl.num_kv_heads, wl.head_dim), device="cuda").to(gb.k_cache.dtype)
    pa.reshape_and_cache(junk, junk, gb.k_cache, gb.v_cache, slots)
    pool.free(intruder)
    in_pairs = pool.swap_in(group[::-1])
    pa.swap_blocks(hk, hv, gb.k_cache, gb.v_cache, torch.from_numpy(in_pairs).cuda())
    tables = np.full_like(gb.tables_np, -1)
    for s in range(wl.num_seqs):
        t = pool.block_table(s)
        tables[s, :len(t)] = t
    assert (tables[group] != gb.tables_np[group]).any()
    gb.tables = torch.from_numpy(tables).cuda()
    after = to_bits(gb.decode())
    assert device_error() == 0
    np.testing.assert_array_equal(after, before)
    kc, vc, otables = oracle_place(wl)
    ref_bits, err = attention.paged_decode_bits(wl.q, kc, vc, otables, wl.context_lens, wl.scale,
                                                wl.block_size, wl.dtype)
    assert not err.any()
    assert max_err(after, ref_bits, wl.dtype) <= TOL[wl.dtype]
