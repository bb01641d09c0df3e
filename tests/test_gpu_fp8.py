"""GPU parity of FP8 (E4M3) KV blocks: the quantising cache write is bit-exact against the
oracle (ties, saturation, subnormals, both scales kinds); paged decode over FP8 blocks is
within the decode tolerance of the oracle's float64 decode over the same codes, for every
head-group shape, head size, block size and query type, bit-identical under physical
block permutations, and flags invalid items; block copies move FP8 blocks exactly."""
import numpy as np
import pytest
import torch

import paged_kv_cache_149_gb300 as pa
import workloads
from gpu_harness import TOL, device_error, max_err, to_bits, to_device
from oracle import fp8
from oracle.block_pool import BlockPool as OraclePool

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(libpa):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    device_error()


def codes(t):
    return t.contiguous().view(torch.uint8).cpu().numpy()


def oracle_place(wl, ks, vs):
    pool = OraclePool(wl.num_blocks, wl.block_size, wl.free_order)
    tables = np.full((wl.num_seqs, wl.max_blocks_per_seq), -1, dtype=np.int32)
    slots = []
    for s in range(wl.num_seqs):
        c = int(wl.context_lens[s])
        pool.allocate(s, c)
        t = pool.block_table(s)
        tables[s, :len(t)] = t
        slots += [pool.slot(s, i) for i in range(c)]
    shape = (wl.num_blocks, wl.num_kv_heads, wl.block_size, wl.head_dim)
    k8, v8 = np.full(shape, 0x7F, np.uint8), np.full(shape, 0x7F, np.uint8)
    return fp8.reshape_and_cache(k8, v8, wl.keys, wl.values, np.array(slots), ks, vs,
                                 wl.dtype) + (tables,)


class Fp8Batch:
    """The library's side: C++ pool tables, K/V quantised into NaN-filled FP8 caches."""

    def __init__(self, wl, ks, vs, free_order=None):
        self.wl, self.ks, self.vs = wl, ks, vs
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
        shape = (wl.num_blocks, wl.num_kv_heads, wl.block_size, wl.head_dim)
        self.k8 = torch.full(shape, 0x7F, dtype=torch.uint8, device="cuda")
        self.v8 = torch.full(shape, 0x7F, dtype=torch.uint8, device="cuda")
        pa.reshape_and_cache_fp8(to_device(wl.keys, wl.dtype), to_device(wl.values, wl.dtype),
                                 self.k8, self.v8, torch.from_numpy(np.concatenate(slots)).cuda(),
                                 ks, vs)
        self.tables_np = tables
        self.tables = torch.from_numpy(tables).cuda()
        self.ctx = torch.from_numpy(wl.context_lens.astype(np.int32)).cuda()
        self.q = to_device(wl.q, wl.dtype)

    def decode(self, tables=None, ctx=None):
        out = pa.decode_fp8(self.q, self.k8, self.v8, self.tables if tables is None else tables,
                            self.ctx if ctx is None else ctx, self.wl.scale, self.ks, self.vs)
        torch.cuda.synchronize()
        return to_bits(out)


def check(wl, ks=0.0123, vs=0.0456, seqs=None):
    gb = Fp8Batch(wl, ks, vs)
    got = gb.decode()
    assert device_error() == 0
    k8, v8, tables = oracle_place(wl, ks, vs)
    np.testing.assert_array_equal(codes(gb.k8), k8)
    np.testing.assert_array_equal(codes(gb.v8), v8)
    np.testing.assert_array_equal(gb.tables_np, tables)
    ref, err = fp8.paged_decode_bits(wl.q, k8, v8, tables, wl.context_lens, wl.scale, ks, vs,
                                     wl.block_size, wl.dtype, seqs=seqs)
    assert not err.any()
    rows = got if seqs is None else got[list(seqs)]
    e = max_err(rows, ref, wl.dtype)
    assert e <= TOL[wl.dtype], f"max abs error {e}"
    return got


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("scale", [2.0 ** -5, 0.0123, 3.7])
def test_cache_write_bit_exact_including_ties_saturation_and_subnormals(dtype, scale):
    rng = np.random.default_rng(int(scale * 1000) + (dtype == "bf16"))
    n, hkv, d, bs, nb = 40, 4, 128, 16, 8
    vals = np.unique(np.abs(fp8.decode_e4m3(np.arange(256, dtype=np.uint8))))
    vals = vals[~np.isnan(vals)]
    mids = (vals[:-1] + vals[1:]) / 2
    special = np.concatenate([vals, mids, -mids, [449, 470, 1e4, -1e4, 2.0 ** -10]]) * scale
    x = rng.standard_normal((n, hkv, d)).astype(np.float32) * 3.0 * scale * 100
    x.reshape(-1)[:len(special)] = special
    key = workloads.to_bits(x, dtype)
    value = workloads.to_bits(x[::-1].copy(), dtype)
    slots = rng.permutation(nb * bs)[:n].astype(np.int64)
    k8 = torch.zeros((nb, hkv, bs, d), dtype=torch.uint8, device="cuda")
    v8 = torch.zeros_like(k8)
    pa.reshape_and_cache_fp8(to_device(key, dtype), to_device(value, dtype), k8, v8,
                             torch.from_numpy(slots).cuda(), scale, scale * 2)
    zero = np.zeros((nb, hkv, bs, d), np.uint8)
    want_k, want_v = fp8.reshape_and_cache(zero, zero, key, value, slots, scale, scale * 2, dtype)
    np.testing.assert_array_equal(codes(k8), want_k)
    np.testing.assert_array_equal(codes(v8), want_v)
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
    wl = workloads.custom("f8", ctx, dtype, hq, hkv, d, bs,
                          sum(-(-c // bs) for c in ctx) + 7, 256, seed=hq * 31 + d + bs)
    check(wl)


def test_one_long_sequence_cut_across_every_cta():
    wl = workloads.custom("f8long", [30000], "bf16", 32, 8, 128, 16, 1900, 30016, seed=3)
    check(wl, ks=0.02, vs=0.03)


def test_llama_batch_every_sequence():
    wl = workloads.llama31_8b()
    check(wl)


def test_permutation_bit_identical():
    wl = workloads.custom("f8p", [100, 33, 700, 5], "bf16", 32, 8, 128, 16, 80, 1024, seed=9)
    a = Fp8Batch(wl, 0.02, 0.03).decode()
    order = np.random.default_rng(2).permutation(wl.num_blocks).astype(np.int32)
    b = Fp8Batch(wl, 0.02, 0.03, free_order=order).decode()
    np.testing.assert_array_equal(a, b)
    assert device_error() == 0


def test_invalid_items_give_zeros_and_flags():
    wl = workloads.custom("f8bad", [20, 40, 60], "fp16", 8, 2, 64, 16, 16, 64, seed=4)
    gb = Fp8Batch(wl, 0.05, 0.05)
    tables = gb.tables_np.copy()
    tables[1, 0] = wl.num_blocks + 3
    ctx = wl.context_lens.astype(np.int32).copy()
    ctx[2] = 0
    got = gb.decode(torch.from_numpy(tables).cuda(), torch.from_numpy(ctx).cuda())
    flags = device_error()
    assert flags == pa.DEVERR_BAD_BLOCK | pa.DEVERR_BAD_CONTEXT
    assert not got[1].any() and not got[2].any() and got[0].any()


def test_fp8_blocks_copy_and_swap_exactly():
    rng = np.random.default_rng(6)
    nb, hkv, bs, d = 24, 8, 16, 128
    k = rng.integers(0, 256, size=(nb, hkv, bs, d), dtype=np.uint8)
    gk, gv = torch.from_numpy(k).cuda(), torch.from_numpy(k[::-1].copy()).cuda()
    pairs = np.array([(0, 10), (3, 11), (3, 12), (23, 13)], dtype=np.int32)
    pa.copy_blocks(gk, gv, torch.from_numpy(pairs).cuda())
    want = k.copy()
    want[pairs[:, 1]] = k[pairs[:, 0]]
    np.testing.assert_array_equal(codes(gk), want)
    hk = torch.zeros((8, hkv, bs, d), dtype=torch.uint8).pin_memory()
    hv = torch.zeros_like(hk).pin_memory()
    sp = np.array([(10, 0), (5, 7)], dtype=np.int32)
    pa.swap_blocks(gk, gv, hk, hv, torch.from_numpy(sp).cuda())
    torch.cuda.synchronize()
    assert np.array_equal(hk.numpy()[0], want[10]) and np.array_equal(hk.numpy()[7], want[5])
    assert device_error() == 0


@pytest.mark.parametrize("recipe", ["tiny", "b8", "llama"])
def test_fused_step_equals_cache_write_then_decode(recipe):
    """pa_decode_append_fp8 quantises each sequence's newest row in the kernel; caches and
    output equal pa_reshape_and_cache_fp8 + pa_decode_fp8 bit for bit."""
    if recipe == "tiny":
        wl = workloads.tiny()
    elif recipe == "b8":
        wl = workloads.custom("f8b8", [1, 8, 9, 16, 17, 33, 200], "bf16", 16, 4, 128, 8,
                              80, 256, seed=12)
    else:
        wl = workloads.llama31_8b(num_seqs=24)
    ks, vs = 0.0123, 0.0234
    outs, caches = [], []
    for fused in (False, True):
        gb = Fp8Batch(wl, ks, vs)   # every token written, the newest included ...
        last = wl.seq_start[1:] - 1
        key_new = to_device(wl.keys[last], wl.dtype)
        value_new = to_device(wl.values[last], wl.dtype)
        # ... then the newest rows' slots poisoned, so only the step can make them right
        slots = np.array([gb.tables_np[s][(int(c) - 1) // wl.block_size] * wl.block_size +
                          (int(c) - 1) % wl.block_size for s, c in enumerate(wl.context_lens)])
        idx = torch.from_numpy(slots).cuda()
        blk, row = idx // wl.block_size, idx % wl.block_size
        gb.k8[blk, :, row] = 0x7F
        gb.v8[blk, :, row] = 0x7F
        if fused:
            out = pa.decode_append_fp8(gb.q, key_new, value_new, gb.k8, gb.v8, gb.tables, gb.ctx,
                                       wl.scale, ks, vs)
        else:
            pa.reshape_and_cache_fp8(key_new, value_new, gb.k8, gb.v8, idx.to(torch.int64), ks, vs)
            out = pa.decode_fp8(gb.q, gb.k8, gb.v8, gb.tables, gb.ctx, wl.scale, ks, vs)
        torch.cuda.synchronize()
        assert device_error() == 0
        outs.append(to_bits(out))
        caches.append((codes(gb.k8), codes(gb.v8)))
    np.testing.assert_array_equal(outs[0], outs[1])
    np.testing.assert_array_equal(caches[0][0], caches[1][0])
    np.testing.assert_array_equal(caches[0][1], caches[1][1])
