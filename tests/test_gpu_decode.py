"""GPU parity of paged decode against the oracle: ragged tails, every GQA group, both
head sizes, all block sizes, both dtypes, cut pairs, and the exact cases."""
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


def check_against_oracle(wl, out_bits):
    """Full oracle (paged, through its own placement) on every sequence."""
    kc, vc, tables = oracle_place(wl)
    ref, err = attention.paged_decode_bits(wl.q, kc, vc, tables, wl.context_lens, wl.scale,
                                           wl.block_size, wl.dtype)
    assert not err.any()
    e = max_err(out_bits, ref, wl.dtype)
    assert e <= TOL[wl.dtype], f"max abs error {e} > {TOL[wl.dtype]}"
    return e


def test_tiny_recipe():
    wl = workloads.tiny()
    gb = GpuBatch(wl)
    out = gb.decode()
    check_against_oracle(wl, to_bits(out))
    assert device_error() == 0


CASES = []
for dtype in ("fp16", "bf16"):
    for d in (64, 128):
        for bs in (8, 16, 32):
            for hq, hkv in ((4, 4), (4, 2), (6, 2), (8, 2), (16, 2), (12, 1)):
                CASES.append((dtype, d, bs, hq, hkv))
# kv-head counts that give every pair-group size (8, 4, 2, 1 pairs per family), several
# families per sequence, and query-head chunks (64 / 2: two chunks of 16)
CASES += [("bf16", 128, 16, 32, 8), ("fp16", 64, 8, 8, 8), ("bf16", 128, 16, 32, 32),
          ("fp16", 128, 32, 24, 12), ("bf16", 64, 16, 12, 6), ("fp16", 128, 16, 6, 3),
          ("bf16", 128, 16, 64, 2), ("fp16", 128, 16, 48, 16)]


@pytest.mark.parametrize("dtype,d,bs,hq,hkv", CASES)
def test_shapes_ragged(dtype, d, bs, hq, hkv):
    ctx = [1, 2, bs - 1, bs, bs + 1, 17, 100, 257, 300, 513]
    T = max(ctx) // bs + 2
    nb = sum(-(-c // bs) for c in ctx) + 7
    seed = CASES.index((dtype, d, bs, hq, hkv))
    wl = workloads.custom("ragged", ctx, dtype, hq, hkv, d, bs, nb, T * bs, seed=seed)
    gb = GpuBatch(wl)
    check_against_oracle(wl, to_bits(gb.decode()))
    assert device_error() == 0


def test_single_token_context_is_exact():
    wl = workloads.custom("one", [1] * 9, "bf16", 32, 8, 128, 16, 16, 64, seed=4)
    gb = GpuBatch(wl)
    out = to_bits(gb.decode())
    v = wl.values.reshape(9, 8, 128)
    for s in range(9):
        for h in range(32):
            np.testing.assert_array_equal(out[s, h], v[s, h // 4])


def test_identical_keys_give_mean_of_values():
    wl = workloads.custom("same", [1000, 37], "fp16", 4, 1, 128, 16, 80, 1024, seed=6)
    wl.keys[:] = wl.keys[0]
    gb = GpuBatch(wl)
    out = formats.decode_bits(to_bits(gb.decode()), "fp16")
    for s in range(2):
        a, b = wl.seq_start[s], wl.seq_start[s + 1]
        mean = formats.decode_bits(wl.values[a:b], "fp16")[:, 0].mean(axis=0)
        for h in range(4):
            assert np.max(np.abs(out[s, h] - mean)) <= TOL["fp16"]


def test_permuting_physical_blocks_is_bit_identical():
    wl = workloads.custom("perm", [5, 700, 1500, 33, 2048, 999], "bf16", 32, 8, 128, 16, 900, 2048, seed=9)
    outs = []
    for seed in (0, 1, 2):
        order = np.random.default_rng(100 + seed).permutation(wl.num_blocks).astype(np.int32)
        gb = GpuBatch(wl, free_order=order)
        outs.append(to_bits(gb.decode()))
    np.testing.assert_array_equal(outs[0], outs[1])
    np.testing.assert_array_equal(outs[0], outs[2])


def test_repeat_calls_are_deterministic():
    wl = workloads.custom("rep", list(range(50, 3000, 97)), "bf16", 32, 8, 128, 16, 3000, 3008, seed=10)
    gb = GpuBatch(wl)
    a = to_bits(gb.decode())
    b = to_bits(gb.decode())
    np.testing.assert_array_equal(a, b)
    check_against_oracle(wl, a)


def test_one_long_sequence_cut_across_every_cta():
    wl = workloads.custom("long1", [40000], "bf16", 8, 2, 128, 16, 2600, 40960, seed=11)
    gb = GpuBatch(wl)
    out = to_bits(gb.decode())
    assert max_err(out[0], oracle_seq_bits(wl, 0), "bf16") <= TOL["bf16"]


def test_invalid_items_give_zeros_and_flags():
    wl = workloads.custom("bad", [20, 5, 40, 7], "fp16", 4, 2, 64, 16, 16, 64, seed=12)
    gb = GpuBatch(wl)
    good = to_bits(gb.decode())
    ctx = gb.ctx.clone()
    ctx[1] = 0
    ctx[3] = 65                        # > T * B = 64
    tables = gb.tables.clone()
    tables[2, 1] = wl.num_blocks + 3    # outside the pool
    out = pa.decode(gb.q, gb.k_cache, gb.v_cache, tables, ctx, wl.scale, workspace=gb.workspace)
    flags = device_error()
    assert flags == pa.DEVERR_BAD_CONTEXT | pa.DEVERR_BAD_BLOCK
    o = to_bits(out)
    assert not o[1].any() and not o[2].any() and not o[3].any()
    np.testing.assert_array_equal(o[0], good[0])


def test_workspace_is_checked():
    wl = workloads.tiny()
    gb = GpuBatch(wl)
    small = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(pa.PagedAttentionError) as e:
        pa.decode(gb.q, gb.k_cache, gb.v_cache, gb.tables, gb.ctx, wl.scale, workspace=small)
    assert e.value.status == pa.PA_ERR_WORKSPACE


def test_misaligned_pointer_is_rejected():
    wl = workloads.tiny()
    gb = GpuBatch(wl)
    flat = torch.empty(gb.q.numel() + 1, dtype=gb.q.dtype, device="cuda")
    q_off = flat[1:].view(gb.q.shape)          # 2-byte offset
    with pytest.raises(pa.PagedAttentionError) as e:
        pa.decode(q_off, gb.k_cache, gb.v_cache, gb.tables, gb.ctx, wl.scale, workspace=gb.workspace)
    assert e.value.status == pa.PA_ERR_ARG


def test_nondefault_stream():
    wl = workloads.custom("stream", [300, 1200], "bf16", 32, 8, 128, 16, 100, 1280, seed=13)
    gb = GpuBatch(wl)
    ref = to_bits(gb.decode())
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        out = gb.decode()
    s.synchronize()
    np.testing.assert_array_equal(to_bits(out), ref)


def test_graph_replays_match_uncaptured_calls():
    """pa_decode captured once in a CUDA graph and replayed with new queries between
    replays gives the same bits as uncaptured calls on those queries.  The long sequence is
    cut across many CTAs, so every replay runs the split-KV merge over the workspace the
    replay before it left behind."""
    wl = workloads.custom("graph", [20000, 300, 4096], "fp16", 8, 2, 128, 16, 1600, 20480, seed=21)
    gb = GpuBatch(wl)
    out = torch.empty_like(gb.q)
    q_in = gb.q.clone()
    gb.decode(out=out)              # first call outside the capture (kernel attributes)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        pa.decode(q_in, gb.k_cache, gb.v_cache, gb.tables, gb.ctx, wl.scale, out=out,
                  workspace=gb.workspace)
    rng = np.random.default_rng(77)
    for _ in range(3):
        q_new = to_device(workloads.normal_bits(rng, wl.q.shape, 1.0, wl.dtype), wl.dtype)
        q_in.copy_(q_new)
        graph.replay()
        torch.cuda.synchronize()
        got = to_bits(out)
        want = to_bits(pa.decode(q_new, gb.k_cache, gb.v_cache, gb.tables, gb.ctx, wl.scale,
                                 workspace=torch.empty_like(gb.workspace)))
        np.testing.assert_array_equal(got, want)
    assert device_error() == 0


@pytest.mark.gpu
def test_timeline_stamps_leave_outputs_unchanged():
    """pa_decode_timeline: the same bits with the stamps on, every warp's three stamps in
    order, and a buffer too small for the grid refused before anything is launched."""
    wl = workloads.custom("timeline", [20000, 300, 4096, 17], "bf16", 32, 8, 128, 16, 1800, 20480,
                          seed=23)
    gb = GpuBatch(wl)
    want = to_bits(gb.decode())
    nsm = torch.cuda.get_device_properties(0).multi_processor_count
    buf = torch.zeros(nsm * 8 * 3, dtype=torch.int64, device="cuda")
    try:
        pa.decode_timeline(buf)
        got = to_bits(gb.decode())
    finally:
        pa.decode_timeline(None)
    np.testing.assert_array_equal(got, want)
    st = buf.view(nsm, 8, 3).cpu().numpy()
    live = st[(st > 0).all(axis=2)]
    assert len(live) >= 8                                   # at least one CTA's warps stamped
    assert (np.diff(live, axis=1) >= 0).all()               # released <= streamed <= end
    small = torch.zeros(8, dtype=torch.int64, device="cuda")
    try:
        pa.decode_timeline(small)
        with pytest.raises(pa.PagedAttentionError):
            gb.decode()
    finally:
        pa.decode_timeline(None)
    assert device_error() == 0
