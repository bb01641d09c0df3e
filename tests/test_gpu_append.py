"""GPU parity of the fused decode step, pa_decode_append: it must leave both caches and the
output bit-identical to pa_reshape_and_cache of each sequence's newest token followed by
pa_decode, and within tolerance of the oracle."""
import ctypes

import numpy as np
import pytest
import torch

import paged_kv_cache_149_gb300 as pa
import workloads
from gpu_harness import (TOL, GpuBatch, device_error, max_err, oracle_place, oracle_seq_bits,
                         to_bits, to_device)
from oracle import attention, formats

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(libpa):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    device_error()


def newest_rows(wl):
    """Each sequence's last logical K and V row, [n, Hkv, d] bit patterns."""
    last = wl.seq_start[1:] - 1
    return wl.keys[last], wl.values[last]


def pre_step(wl):
    """The library's placement of the whole batch, then each sequence's newest slot put back
    to NaN: the caches as they are before the step writes its tokens."""
    gb = GpuBatch(wl)
    slots = np.array([gb.pool.slots(s, int(wl.context_lens[i]) - 1, 1)[0]
                      for i, s in enumerate(gb.seq_ids)], dtype=np.int64)
    blk = torch.from_numpy(slots // wl.block_size).cuda()
    row = torch.from_numpy(slots % wl.block_size).cuda()
    nan = int(np.uint16(formats.FORMATS[wl.dtype]["qnan"]).view(np.int16))
    for c in (gb.k_cache, gb.v_cache):
        c.view(torch.int16)[blk, :, row, :] = nan
    return gb, torch.from_numpy(slots).cuda()


def both_paths(wl):
    gb, slots = pre_step(wl)
    kn, vn = newest_rows(wl)
    kn, vn = to_device(kn, wl.dtype), to_device(vn, wl.dtype)
    k_a, v_a = gb.k_cache.clone(), gb.v_cache.clone()
    pa.reshape_and_cache(kn, vn, k_a, v_a, slots)
    out_a = pa.decode(gb.q, k_a, v_a, gb.tables, gb.ctx, wl.scale, workspace=gb.workspace)
    k_b, v_b = gb.k_cache.clone(), gb.v_cache.clone()
    out_b = pa.decode_append(gb.q, kn, vn, k_b, v_b, gb.tables, gb.ctx, wl.scale,
                             workspace=gb.workspace)
    torch.cuda.synchronize()
    return (to_bits(out_a), to_bits(k_a), to_bits(v_a)), (to_bits(out_b), to_bits(k_b), to_bits(v_b))


def check(wl, oracle_seqs=None):
    a, b = both_paths(wl)
    for x, y, what in zip(a, b, ("out", "k_cache", "v_cache")):
        np.testing.assert_array_equal(x, y, err_msg=what)
    assert device_error() == 0
    if oracle_seqs is None:  # the full oracle, through its own placement
        kc, vc, tables = oracle_place(wl)
        ref, err = attention.paged_decode_bits(wl.q, kc, vc, tables, wl.context_lens, wl.scale,
                                               wl.block_size, wl.dtype)
        assert not err.any()
        e = max_err(a[0], ref, wl.dtype)
    else:  # sampled sequences, from their logical rows
        e = max(max_err(a[0][s], oracle_seq_bits(wl, s), wl.dtype) for s in oracle_seqs)
    assert e <= TOL[wl.dtype], f"max abs error {e}"


def test_tiny():
    check(workloads.tiny())


# every pair-group size (8, 4, 2, 1 pairs per family), both head sizes, all block sizes
SHAPES = [("bf16", 128, 16, 32, 8), ("fp16", 64, 8, 8, 2), ("bf16", 128, 32, 6, 3),
          ("fp16", 128, 16, 32, 32), ("bf16", 64, 16, 24, 12), ("fp16", 128, 8, 16, 16)]


@pytest.mark.parametrize("dtype,d,bs,hq,hkv", SHAPES)
def test_shapes(dtype, d, bs, hq, hkv):
    ctx = [1, 2, bs - 1, bs, bs + 1, 17, 100, 257, 300, 513]
    T = max(ctx) // bs + 2
    nb = sum(-(-c // bs) for c in ctx) + 7
    wl = workloads.custom("append", ctx, dtype, hq, hkv, d, bs, nb, T * bs, seed=SHAPES.index(
        (dtype, d, bs, hq, hkv)) + 40)
    check(wl)


def test_long_sequence_cut_across_every_cta():
    wl = workloads.custom("append_long", [40000], "bf16", 8, 2, 128, 16, 2600, 40960, seed=51)
    check(wl)


def test_llama31_8b_batch():
    check(workloads.llama31_8b(), oracle_seqs=range(0, 64, 9))


def test_invalid_context_writes_nothing():
    wl = workloads.custom("append_bad", [20, 33, 5], "bf16", 8, 2, 64, 16, 12, 64, seed=52)
    gb, _ = pre_step(wl)
    kn, vn = newest_rows(wl)
    kn, vn = to_device(kn, wl.dtype), to_device(vn, wl.dtype)
    ctx = gb.ctx.clone()
    ctx[1] = 0
    k0, v0 = to_bits(gb.k_cache), to_bits(gb.v_cache)
    out = pa.decode_append(gb.q, kn, vn, gb.k_cache, gb.v_cache, gb.tables, ctx, wl.scale,
                           workspace=gb.workspace)
    flags = device_error()
    assert flags & 0x2  # PA_DEVERR_BAD_CONTEXT
    assert not to_bits(out[1]).any()
    # sequence 1 wrote nothing; 0 and 2 wrote their newest rows
    kc = to_bits(gb.k_cache)
    changed = np.argwhere((kc != k0).any(axis=(1, 3)))
    s0 = gb.pool.slots(gb.seq_ids[0], 19, 1)[0]
    s2 = gb.pool.slots(gb.seq_ids[2], 4, 1)[0]
    assert sorted(map(tuple, changed)) == sorted([(s0 // 16, s0 % 16), (s2 // 16, s2 % 16)])
    assert (to_bits(gb.v_cache) != v0).any()


def test_missing_new_rows_is_an_argument_error():
    wl = workloads.tiny()
    gb = GpuBatch(wl)
    n, hq, d = gb.q.shape
    nb, hkv, bs, _ = gb.k_cache.shape
    ws = gb.workspace
    st = pa.lib().pa_decode_append(
        gb.q.data_ptr(), None, None, gb.k_cache.data_ptr(), gb.v_cache.data_ptr(),
        gb.tables.data_ptr(), gb.tables.shape[1], gb.ctx.data_ptr(), n, hq, hkv, d, bs, nb,
        ctypes.c_float(wl.scale), torch.empty_like(gb.q).data_ptr(), ws.data_ptr(),
        ws.numel() * ws.element_size(), 0 if wl.dtype == "fp16" else 1, None)
    assert st == -1  # PA_ERR_ARG


@pytest.mark.parametrize("fmt", ["16", "fp8", "int4"])
def test_planned_launch_equals_the_call(fmt):
    """A Launch planned once (plan=True) and run on a stream gives the same output and
    caches as the plain call, for every block format."""
    wl = workloads.llama31_8b(num_seqs=12)
    kn, vn = (to_device(x, wl.dtype) for x in newest_rows(wl))
    stream = torch.cuda.Stream()
    results = []
    for planned in (False, True):
        if fmt == "16":
            gb, _ = pre_step(wl)
            caches = (gb.k_cache, gb.v_cache)
            call = lambda **kw: pa.decode_append(gb.q, kn, vn, gb.k_cache, gb.v_cache, gb.tables,
                                                 gb.ctx, wl.scale, **kw)
        else:
            from test_gpu_fp8 import Fp8Batch
            from test_gpu_int4 import Int4Batch
            gb = Fp8Batch(wl, 0.0123, 0.0234) if fmt == "fp8" else Int4Batch(wl)
            if fmt == "fp8":
                caches = (gb.k8, gb.v8)
                call = lambda **kw: pa.decode_append_fp8(gb.q, kn, vn, gb.k8, gb.v8, gb.tables,
                                                         gb.ctx, wl.scale, 0.0123, 0.0234, **kw)
            else:
                caches = (gb.kc, gb.vc, gb.ks.view(torch.int32), gb.vs.view(torch.int32))
                call = lambda **kw: pa.decode_append_int4(gb.q, kn, vn, gb.kc, gb.vc, gb.ks, gb.vs,
                                                          gb.tables, gb.ctx, wl.scale, **kw)
        out = torch.empty((wl.num_seqs, wl.num_q_heads, wl.head_dim), dtype=kn.dtype, device="cuda")
        torch.cuda.synchronize()  # the caches were built on the default stream
        if planned:
            launch = call(out=out, plan=True)
            launch.run(stream)
            launch.run(stream)  # a second run over the same buffers gives the same result
        else:
            call(out=out, stream=stream)
        stream.synchronize()
        assert device_error() == 0
        results.append([to_bits(out)] + [c.contiguous().view(torch.uint8).cpu().numpy() for c in caches])
    for a, b in zip(*results):
        np.testing.assert_array_equal(a, b)
