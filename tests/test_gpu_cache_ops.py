"""GPU parity of the cache write and the block copy: bit-exact against the oracle."""
import numpy as np
import pytest
import torch

import workloads
from gpu_harness import GpuBatch, nan_cache, oracle_place, to_bits, to_device, device_error
from oracle import cache_ops

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(libpa):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    device_error()  # clear the word


@pytest.mark.parametrize("recipe", ["tiny", "b8", "b32_d128"])
def test_placement_tables_and_caches_bit_exact(recipe):
    if recipe == "tiny":
        wl = workloads.tiny()
    elif recipe == "b8":
        wl = workloads.custom("b8", [1, 8, 9, 31, 64, 65], "bf16", 6, 3, 64, 8, 64, 72, seed=2)
    else:
        wl = workloads.custom("b32", [3, 32, 33, 95, 200], "fp16", 8, 2, 128, 32, 40, 224, seed=3)
    gb = GpuBatch(wl)
    kc, vc, tables = oracle_place(wl)
    np.testing.assert_array_equal(gb.tables_np, tables)
    np.testing.assert_array_equal(to_bits(gb.k_cache), kc)
    np.testing.assert_array_equal(to_bits(gb.v_cache), vc)
    assert device_error() == 0


def test_reshape_skips_negative_and_flags_out_of_pool():
    rng = np.random.default_rng(5)
    nb, hkv, bs, d = 6, 2, 16, 64
    key = rng.integers(0, 30000, size=(5, hkv, d), dtype=np.uint16)
    val = rng.integers(0, 30000, size=(5, hkv, d), dtype=np.uint16)
    slots = np.array([3, -1, 95, nb * bs, 17], dtype=np.int64)  # 96 is outside the pool
    kc = nan_cache(nb, hkv, bs, d, "fp16")
    vc = nan_cache(nb, hkv, bs, d, "fp16")
    import paged_kv_cache_149_gb300 as pa
    pa.reshape_and_cache(to_device(key, "fp16"), to_device(val, "fp16"), kc, vc,
                         torch.from_numpy(slots).cuda())
    assert device_error() == pa.DEVERR_BAD_SLOT
    ok = slots.copy()
    ok[3] = -1
    k0 = to_bits(nan_cache(nb, hkv, bs, d, "fp16"))
    want_k, want_v = cache_ops.reshape_and_cache(k0, k0.copy(), key, val, ok)
    np.testing.assert_array_equal(to_bits(kc), want_k)
    np.testing.assert_array_equal(to_bits(vc), want_v)


@pytest.mark.parametrize("dtype,d,bs", [("bf16", 128, 16), ("fp16", 64, 8), ("bf16", 64, 32)])
def test_copy_blocks_bit_exact(dtype, d, bs):
    import paged_kv_cache_149_gb300 as pa
    rng = np.random.default_rng(7)
    nb, hkv = 40, 8
    kc = rng.integers(0, 65535, size=(nb, hkv, bs, d), dtype=np.uint16)
    vc = rng.integers(0, 65535, size=(nb, hkv, bs, d), dtype=np.uint16)
    pairs = [(0, 20), (5, 21), (5, 22), (39, 23), (1, 24)]
    pa.check_block_mapping(pairs, nb)
    gk, gv = to_device(kc, dtype), to_device(vc, dtype)
    pa.copy_blocks(gk, gv, torch.tensor(pairs, dtype=torch.int32, device="cuda"))
    want_k, want_v = cache_ops.copy_blocks(kc, vc, pairs)
    np.testing.assert_array_equal(to_bits(gk), want_k)
    np.testing.assert_array_equal(to_bits(gv), want_v)
    assert device_error() == 0


def test_copy_blocks_flags_bad_ids():
    import paged_kv_cache_149_gb300 as pa
    rng = np.random.default_rng(8)
    kc = rng.integers(0, 65535, size=(8, 2, 16, 64), dtype=np.uint16)
    gk, gv = to_device(kc, "fp16"), to_device(kc, "fp16")
    pa.copy_blocks(gk, gv, torch.tensor([(0, 5), (9, 6), (1, -2)], dtype=torch.int32, device="cuda"))
    assert device_error() == pa.DEVERR_BAD_PAIR
    want, _ = cache_ops.copy_blocks(kc, kc, [(0, 5)])
    np.testing.assert_array_equal(to_bits(gk), want)
