"""GPU parity of INT4 KV blocks (4-bit codes with a float32 scale per row): the quantising
cache write is bit-exact against the oracle (codes and scales; ties, zero rows, wide
magnitudes); paged decode over INT4 blocks is within the decode tolerance of the oracle's
float64 decode over the same codes and scales, for every head-group shape, head size,
block size and query type, bit-identical under physical block permutations, and flags
invalid items; the fused step equals write + decode bit for bit; block copies and swaps
move codes and scales exactly."""
import numpy as np
import pytest
import torch

import paged_kv_cache_149_gb300 as pa
import workloads
from gpu_harness import TOL, device_error, max_err, to_bits, to_device
from oracle import int4
from oracle.block_pool import BlockPool as OraclePool

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(libpa):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    device_error()


def np_(t):
    return t.contiguous().cpu().numpy()


def oracle_place(wl):
    pool = OraclePool(wl.num_blocks, wl.block_size, wl.free_order)
    tables = np.full((wl.num_seqs, wl.max_blocks_per_seq), -1, dtype=np.int32)
    slots = []
    for s in range(wl.num_seqs):
        c = int(wl.context_lens[s])
        pool.allocate(s, c)
        t = pool.block_table(s)
        tables[s, :len(t)] = t
        slots += [pool.slot(s, i) for i in range(c)]
    nb, hkv, b, d = wl.num_blocks, wl.num_kv_heads, wl.block_size, wl.head_dim
    kc = np.full((nb, hkv, b, d // 2), 0xFF, np.uint8)
    ks = np.full((nb, hkv, b), np.nan, np.float32)
    return int4.reshape_and_cache(kc, kc.copy(), ks, ks.copy(), wl.keys, wl.values, np.array(slots),
                                  wl.dtype) + (tables,)


class Int4Batch:
    """The library's side: C++ pool tables, K/V quantised into garbage-filled INT4 caches
    (codes 0xFF, scales NaN: nothing outside the contexts may be read)."""

    def __init__(self, wl, free_order=None):
        self.wl = wl
        order = wl.free_order if free_order is None else free_order
        pool = pa.BlockPool(wl.num_blocks, wl.block_size, order)
        tables = np.full((wl.num_seqs, wl.max_blocks_per_seq), -1, dtype=np.int32)
        slots = []
        for s in range(wl.num_seqs):
            c = int(wl.context_lens[s])
            pool.allocate(s, c)
            t = pool.block_table(s)
            tables[s, :len(t)] = t
            slots.append(pool.slots(s, 0, c))
        nb, hkv, b, d = wl.num_blocks, wl.num_kv_heads, wl.block_size, wl.head_dim
        self.kc = torch.full((nb, hkv, b, d // 2), 0xFF, dtype=torch.uint8, device="cuda")
        self.vc = torch.full_like(self.kc, 0xFF)
        self.ks = torch.full((nb, hkv, b), float("nan"), dtype=torch.float32, device="cuda")
        self.vs = torch.full_like(self.ks, float("nan"))
        pa.reshape_and_cache_int4(to_device(wl.keys, wl.dtype), to_device(wl.values, wl.dtype),
                                  self.kc, self.vc, self.ks, self.vs,
                                  torch.from_numpy(np.concatenate(slots)).cuda())
        self.tables_np = tables
        self.tables = torch.from_numpy(tables).cuda()
        self.ctx = torch.from_numpy(wl.context_lens.astype(np.int32)).cuda()
        self.q = to_device(wl.q, wl.dtype)

    def decode(self, tables=None, ctx=None):
        out = pa.decode_int4(self.q, self.kc, self.vc, self.ks, self.vs,
                             self.tables if tables is None else tables,
                             self.ctx if ctx is None else ctx, self.wl.scale)
        torch.cuda.synchronize()
        return to_bits(out)


def same_caches(gb, want):
    kc, vc, ks, vs = want[:4]
    np.testing.assert_array_equal(np_(gb.kc), kc)
    np.testing.assert_array_equal(np_(gb.vc), vc)
    # float32 scales compared as bit patterns (NaN where nothing was written)
    np.testing.assert_array_equal(np_(gb.ks).view(np.uint32), ks.view(np.uint32))
    np.testing.assert_array_equal(np_(gb.vs).view(np.uint32), vs.view(np.uint32))


def check(wl, seqs=None):
    gb = Int4Batch(wl)
    got = gb.decode()
    assert device_error() == 0
    want = oracle_place(wl)
    same_caches(gb, want)
    np.testing.assert_array_equal(gb.tables_np, want[4])
    ref, err = int4.paged_decode_bits(wl.q, *want[:4], want[4], wl.context_lens, wl.scale,
                                      wl.block_size, wl.dtype, seqs=seqs)
    assert not err.any()
    rows = got if seqs is None else got[list(seqs)]
    e = max_err(rows, ref, wl.dtype)
    assert e <= TOL[wl.dtype], f"max abs error {e}"
    return got


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("d", [64, 128])
def test_cache_write_bit_exact_including_ties_zero_rows_and_wide_magnitudes(dtype, d):
    rng = np.random.default_rng(d + (dtype == "bf16"))
    n, hkv, bs, nb = 48, 4, 16, 8
    x = rng.standard_normal((n, hkv, d)).astype(np.float32) * rng.uniform(1e-3, 50, (n, hkv, 1))
    # rows with max |x| = 7 * 2^k (s = 2^k exactly) and halves in between: exact ties
    for r in range(6):
        k = float(2.0 ** (r - 3))
        row = rng.integers(-14, 15, size=d) / 2.0
        row[0] = 7.0
        x[r, r % hkv] = (row * k).astype(np.float32)
    x[7, :] = 0.0                       # all-zero rows
    x[8, 1, :] = 0.0
    x[8, 1, 5] = -1e-4                  # a single tiny value
    key = workloads.to_bits(x, dtype)
    value = workloads.to_bits(x[::-1].copy(), dtype)
    slots = rng.permutation(nb * bs)[:n].astype(np.int64)
    kc = torch.zeros((nb, hkv, bs, d // 2), dtype=torch.uint8, device="cuda")
    vc = torch.zeros_like(kc)
    ks = torch.zeros((nb, hkv, bs), dtype=torch.float32, device="cuda")
    vs = torch.zeros_like(ks)
    pa.reshape_and_cache_int4(to_device(key, dtype), to_device(value, dtype), kc, vc, ks, vs,
                              torch.from_numpy(slots).cuda())
    zc = np.zeros((nb, hkv, bs, d // 2), np.uint8)
    zs = np.zeros((nb, hkv, bs), np.float32)
    want = int4.reshape_and_cache(zc, zc, zs, zs, key, value, slots, dtype)
    np.testing.assert_array_equal(np_(kc), want[0])
    np.testing.assert_array_equal(np_(vc), want[1])
    np.testing.assert_array_equal(np_(ks).view(np.uint32), want[2].view(np.uint32))
    np.testing.assert_array_equal(np_(vs).view(np.uint32), want[3].view(np.uint32))
    assert device_error() == 0


def test_tiny():
    check(workloads.tiny())


CASES = []
for dtype in ("fp16", "bf16"):
    for d in (64, 128):
        for bs in (8, 16, 32):
            for hq, hkv in ((4, 4), (8, 2), (12, 4), (32, 8), (32, 2), (64, 4), (6, 3)):
                CASES.append((dtype, d, bs, hq, hkv))


@pytest.mark.parametrize("dtype,d,bs,hq,hkv", CASES)
def test_shapes_ragged(dtype, d, bs, hq, hkv):
    ctx = [1, bs - 1, bs, bs + 1, 3 * bs + 5, 200, 17, 64]
    wl = workloads.custom("i4", ctx, dtype, hq, hkv, d, bs,
                          sum(-(-c // bs) for c in ctx) + 7, 256, seed=hq * 31 + d + bs)
    check(wl)


def test_one_long_sequence_cut_across_every_cta():
    wl = workloads.custom("i4long", [30000], "bf16", 32, 8, 128, 16, 1900, 30016, seed=3)
    check(wl)


def test_llama_batch_every_sequence():
    wl = workloads.llama31_8b()
    check(wl)


def test_permutation_bit_identical():
    wl = workloads.custom("i4p", [100, 33, 700, 5], "bf16", 32, 8, 128, 16, 80, 1024, seed=9)
    a = Int4Batch(wl).decode()
    order = np.random.default_rng(2).permutation(wl.num_blocks).astype(np.int32)
    b = Int4Batch(wl, free_order=order).decode()
    np.testing.assert_array_equal(a, b)
    assert device_error() == 0


def test_invalid_items_give_zeros_and_flags():
    wl = workloads.custom("i4bad", [20, 40, 60], "fp16", 8, 2, 64, 16, 16, 64, seed=4)
    gb = Int4Batch(wl)
    tables = gb.tables_np.copy()
    tables[1, 0] = wl.num_blocks + 3
    ctx = wl.context_lens.astype(np.int32).copy()
    ctx[2] = 0
    got = gb.decode(torch.from_numpy(tables).cuda(), torch.from_numpy(ctx).cuda())
    assert device_error() == pa.DEVERR_BAD_BLOCK | pa.DEVERR_BAD_CONTEXT
    assert not got[1].any() and not got[2].any() and got[0].any()


@pytest.mark.parametrize("recipe", ["tiny", "b8", "llama"])
def test_fused_step_equals_cache_write_then_decode(recipe):
    if recipe == "tiny":
        wl = workloads.tiny()
    elif recipe == "b8":
        wl = workloads.custom("i4b8", [1, 8, 9, 16, 17, 33, 200], "bf16", 16, 4, 128, 8, 80, 256,
                              seed=12)
    else:
        wl = workloads.llama31_8b(num_seqs=24)
    outs, caches = [], []
    for fused in (False, True):
        gb = Int4Batch(wl)
        last = wl.seq_start[1:] - 1
        key_new = to_device(wl.keys[last], wl.dtype)
        value_new = to_device(wl.values[last], wl.dtype)
        slots = np.array([gb.tables_np[s][(int(c) - 1) // wl.block_size] * wl.block_size +
                          (int(c) - 1) % wl.block_size for s, c in enumerate(wl.context_lens)])
        idx = torch.from_numpy(slots).cuda()
        blk, row = idx // wl.block_size, idx % wl.block_size
        gb.kc[blk, :, row] = 0xFF          # the newest rows poisoned: only the step fixes them
        gb.vc[blk, :, row] = 0xFF
        gb.ks[blk, :, row] = float("nan")
        gb.vs[blk, :, row] = float("nan")
        if fused:
            out = pa.decode_append_int4(gb.q, key_new, value_new, gb.kc, gb.vc, gb.ks, gb.vs,
                                        gb.tables, gb.ctx, wl.scale)
        else:
            pa.reshape_and_cache_int4(key_new, value_new, gb.kc, gb.vc, gb.ks, gb.vs,
                                      idx.to(torch.int64))
            out = pa.decode_int4(gb.q, gb.kc, gb.vc, gb.ks, gb.vs, gb.tables, gb.ctx, wl.scale)
        torch.cuda.synchronize()
        assert device_error() == 0
        outs.append(to_bits(out))
        caches.append([np_(t) for t in (gb.kc, gb.vc, gb.ks.view(torch.int32), gb.vs.view(torch.int32))])
    np.testing.assert_array_equal(outs[0], outs[1])
    for a, b in zip(*caches):
        np.testing.assert_array_equal(a, b)


def test_int4_blocks_copy_and_swap_exactly():
    rng = np.random.default_rng(6)
    nb, hkv, bs, d = 24, 8, 16, 128
    kc = rng.integers(0, 256, size=(nb, hkv, bs, d // 2), dtype=np.uint8)
    ks = rng.standard_normal((nb, hkv, bs)).astype(np.float32)
    g = [torch.from_numpy(a).cuda() for a in (kc, kc[::-1].copy(), ks, ks[::-1].copy())]
    pairs = np.array([(0, 10), (3, 11), (3, 12), (23, 13)], dtype=np.int32)
    pa.copy_blocks_int4(*g, torch.from_numpy(pairs).cuda())
    want_c, want_s = kc.copy(), ks.copy()
    want_c[pairs[:, 1]] = kc[pairs[:, 0]]
    want_s[pairs[:, 1]] = ks[pairs[:, 0]]
    np.testing.assert_array_equal(np_(g[0]), want_c)
    np.testing.assert_array_equal(np_(g[2]), want_s)
    host = [torch.zeros((8,) + t.shape[1:], dtype=t.dtype).pin_memory() for t in g]
    sp = np.array([(10, 0), (5, 7)], dtype=np.int32)
    pa.swap_blocks_int4(g, host, torch.from_numpy(sp).cuda())
    torch.cuda.synchronize()
    assert np.array_equal(host[0].numpy()[0], want_c[10]) and np.array_equal(host[0].numpy()[7], want_c[5])
    assert np.array_equal(host[2].numpy()[0], want_s[10]) and np.array_equal(host[3].numpy()[7], np_(g[3])[5])
    assert device_error() == 0
