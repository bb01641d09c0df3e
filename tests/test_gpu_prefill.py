"""GPU parity of paged prefill against the oracle: prompts from scratch and chunks, ragged
lengths, every GQA group shape the kernel packs (G = 1..64, with and without a remainder
of rows), both head sizes, all block sizes, both dtypes; physical-block permutations
(bit-identical); invalid items; the benchmark batches, every row; score ranges whose row
maximum grows by more than 2^8 (in exp2 units) from one key tile to the next."""
import numpy as np
import pytest
import torch

import paged_kv_cache_149_gb300 as pa
import workloads
from gpu_harness import TOL, GpuBatch, device_error, max_err, oracle_place, to_bits
from oracle import prefill as oracle_prefill

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(libpa):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    device_error()


def run_gpu(wl, free_order=None, ctx=None, tables=None):
    gb = GpuBatch(wl, free_order=free_order)
    qs = torch.from_numpy(wl.query_start.astype(np.int32)).cuda()
    qlen = np.diff(wl.query_start)
    out = pa.prefill(gb.q, gb.k_cache, gb.v_cache, gb.tables if tables is None else tables,
                     gb.ctx if ctx is None else ctx, qs, wl.scale, int(qlen.max()))
    torch.cuda.synchronize()
    return gb, to_bits(out)


def check(wl, seqs=None):
    gb, got = run_gpu(wl)
    assert device_error() == 0
    kc, vc, tables = oracle_place(wl)
    ref, err = oracle_prefill.paged_prefill_bits(wl.q, kc, vc, tables, wl.context_lens,
                                                 wl.query_start, wl.scale, wl.block_size,
                                                 wl.dtype, seqs=seqs)
    assert not err.any()
    rows = (np.concatenate([np.arange(wl.query_start[s], wl.query_start[s + 1]) for s in seqs])
            if seqs is not None else slice(None))
    e = max_err(got[rows], ref[rows], wl.dtype)
    assert e <= TOL[wl.dtype], f"max abs error {e}"
    return got


def test_tiny():
    check(workloads.prefill_tiny())


CASES = []
for dtype in ("fp16", "bf16"):
    for d in (64, 128):
        for bs in (8, 16, 32):
            for hq, hkv in ((4, 4), (8, 2), (12, 4), (32, 8), (64, 1), (6, 2)):
                CASES.append((dtype, d, bs, hq, hkv))


@pytest.mark.parametrize("dtype,d,bs,hq,hkv", CASES)
def test_shapes_ragged(dtype, d, bs, hq, hkv):
    ctx = [1, 15, 16, 17, 64, 65, 130, 200]
    qlen = [1, 15, 16, 5, 64, 20, 130, 77]
    T = max(ctx) // bs + 2
    nb = sum(-(-c // bs) for c in ctx) + 7
    seed = CASES.index((dtype, d, bs, hq, hkv))
    rng = np.random.default_rng(seed)
    wl = workloads._prefill("ragged", rng, ctx, qlen, dtype, hq, hkv, d, bs, nb, T * bs,
                            1.0 / np.sqrt(d))
    check(wl)


def test_physical_block_permutation_is_bit_identical():
    rng = np.random.default_rng(60)
    wl = workloads._prefill("perm", rng, [300, 77, 513], [300, 40, 129], "bf16", 32, 8, 128,
                            16, 80, 528, 1.0 / np.sqrt(128))
    outs = []
    for seed in (0, 1, 2):
        order = np.random.default_rng(200 + seed).permutation(wl.num_blocks).astype(np.int32)
        outs.append(run_gpu(wl, free_order=order)[1])
    np.testing.assert_array_equal(outs[0], outs[1])
    np.testing.assert_array_equal(outs[0], outs[2])


def test_invalid_items_give_zeros_and_flags():
    wl = workloads.prefill_tiny()
    gb = GpuBatch(wl)
    ctx = gb.ctx.clone()
    ctx[0] = 3                                  # q_len 5 > ctx 3
    tables = gb.tables.clone()
    tables[1, 0] = wl.num_blocks                # a bad block id in sequence 1
    qs = torch.from_numpy(wl.query_start.astype(np.int32)).cuda()
    out = pa.prefill(gb.q, gb.k_cache, gb.v_cache, tables, ctx, qs, wl.scale, 33)
    flags = device_error()
    assert flags & 0x2 and flags & 0x1
    got = to_bits(out)
    assert not got[:wl.query_start[2]].any()
    kc, vc, t_or = oracle_place(wl)
    ref, _ = oracle_prefill.paged_prefill_bits(wl.q, kc, vc, t_or, wl.context_lens,
                                               wl.query_start, wl.scale, wl.block_size,
                                               wl.dtype, seqs=[2, 3])
    assert max_err(got[wl.query_start[2]:], ref[wl.query_start[2]:], wl.dtype) <= TOL[wl.dtype]


def test_chunked_batch_every_sequence():
    """The benchmark's chunked batch (16 chunks of 512 over 1-4 K contexts), every row."""
    check(workloads.prefill_chunked())


def test_prompts_from_scratch_every_sequence():
    """The benchmark's batch of 8 prompts of 2048 tokens from scratch, every row."""
    check(workloads.prefill_llama31_8b())


def test_planned_launches_match_direct_calls():
    """plan=True: a Launch marshalled once writes the same cache rows and the same outputs,
    bit for bit, as the direct calls, and each run reads what the buffers hold then."""
    rng = np.random.default_rng(61)
    wl = workloads._prefill("plan", rng, [300, 77, 513], [300, 40, 129], "bf16", 32, 8, 128,
                            16, 80, 528, 1.0 / np.sqrt(128))
    gb = GpuBatch(wl)
    qs = torch.from_numpy(wl.query_start.astype(np.int32)).cuda()
    maxq = int(np.diff(wl.query_start).max())
    n_new = int(wl.query_start[-1])
    g = torch.Generator(device="cuda").manual_seed(7)
    kn = torch.randn((n_new, wl.num_kv_heads, wl.head_dim), generator=g, device="cuda").to(gb.q.dtype)
    vn = torch.randn(kn.shape, generator=g, device="cuda").to(gb.q.dtype)
    slots = []
    for s in range(wl.num_seqs):
        c, ql = int(wl.context_lens[s]), int(wl.query_start[s + 1] - wl.query_start[s])
        row = gb.tables[s].cpu().numpy()
        for t in range(c - ql, c):
            slots.append(int(row[t // wl.block_size]) * wl.block_size + t % wl.block_size)
    slots = torch.tensor(slots, dtype=torch.int64, device="cuda")
    kc0, vc0 = gb.k_cache.clone(), gb.v_cache.clone()
    stream = torch.cuda.Stream()
    torch.cuda.synchronize()  # (the batch was set up on the default stream)

    pa.reshape_and_cache(kn, vn, gb.k_cache, gb.v_cache, slots, stream=stream)
    want = pa.prefill(gb.q, gb.k_cache, gb.v_cache, gb.tables, gb.ctx, qs, wl.scale, maxq,
                      stream=stream)
    stream.synchronize()
    want_k, want_v, want = gb.k_cache.clone(), gb.v_cache.clone(), want.clone()

    gb.k_cache.copy_(kc0)
    gb.v_cache.copy_(vc0)
    out = torch.empty_like(gb.q)
    w = pa.reshape_and_cache(kn, vn, gb.k_cache, gb.v_cache, slots, plan=True)
    pf = pa.prefill(gb.q, gb.k_cache, gb.v_cache, gb.tables, gb.ctx, qs, wl.scale, maxq,
                    out=out, plan=True)
    torch.cuda.synchronize()
    w.run(stream)
    pf.run(stream)
    stream.synchronize()
    bits = lambda t: t.view(torch.int16)  # (unused cache slots hold NaN)
    assert torch.equal(bits(gb.k_cache), bits(want_k)) and torch.equal(bits(gb.v_cache), bits(want_v))
    assert torch.equal(bits(out), bits(want))
    # a later run reads the buffers' new contents
    gb.q.mul_(-1)
    torch.cuda.synchronize()
    pf.run(stream)
    direct = pa.prefill(gb.q, gb.k_cache, gb.v_cache, gb.tables, gb.ctx, qs, wl.scale, maxq,
                        stream=stream)
    stream.synchronize()
    assert torch.equal(bits(out), bits(direct)) and not torch.equal(bits(out), bits(want))
    assert device_error() == 0
