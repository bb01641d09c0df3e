"""GPU parity where the softmax is far from flat: a key aligned with the query that takes
nearly all the weight, keys drawn with a large spread (scores spanning tens of units),
and scores rising along the context so that the running maximum grows at every stage and
across the pieces of pairs cut between CTAs; for prefill, scores rising fast enough that
a row's maximum grows by more than 2^8 (in exp2 units) from one 64-key tile to the next.
The inputs are shaped here; the oracle and the kernels see only their bits."""
import math

import numpy as np
import pytest
import torch

import paged_kv_cache_149_gb300 as pa
import workloads
from gpu_harness import TOL, GpuBatch, device_error, max_err, oracle_place, oracle_seq_bits, to_bits
from oracle import formats
from oracle import prefill as oracle_prefill

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(libpa):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    device_error()


def as_float(bits, dtype):
    return formats.decode_bits(bits, dtype).astype(np.float32)


def every_sequence_error(wl, out_bits):
    return max(max_err(out_bits[s], oracle_seq_bits(wl, s), wl.dtype) for s in range(wl.num_seqs))


SHAPES = [("bf16", 32, 8), ("fp16", 32, 8), ("fp16", 32, 32), ("bf16", 8, 2)]
CTX = [1, 17, 300, 2049, 9000]


def batch(dtype, hq, hkv, seed, k_std=1.0):
    """K ~ N(0, k_std^2), V ~ N(0, 1)."""
    T = max(CTX) // 16 + 1
    nb = sum(-(-c // 16) for c in CTX) + 5
    wl = workloads.custom("peaked", CTX, dtype, hq, hkv, 128, 16, nb, T * 16, seed=seed)
    if k_std != 1.0:
        wl.keys = workloads.to_bits(as_float(wl.keys, dtype) * np.float32(k_std), dtype)
    return wl


@pytest.mark.parametrize("dtype,hq,hkv", SHAPES)
def test_one_hot_key_takes_the_weight(dtype, hq, hkv):
    """For every sequence and kv head, one key is set to c * q of the group's first head,
    with c chosen so that head's score there is 40 (softmax weight about 1 - e^-35)."""
    wl = batch(dtype, hq, hkv, seed=SHAPES.index((dtype, hq, hkv)))
    g = hq // hkv
    keys = as_float(wl.keys, dtype)
    q = as_float(wl.q, dtype).astype(np.float64)
    rng = np.random.default_rng(5)
    picks = {}
    for s in range(wl.num_seqs):
        a, c = int(wl.seq_start[s]), int(wl.context_lens[s])
        for kvh in range(hkv):
            t = int(rng.integers(0, c))
            qh = q[s, kvh * g]
            keys[a + t, kvh] = (40.0 / (wl.scale * float(qh @ qh))) * qh
            picks[(s, kvh)] = a + t
    wl.keys = workloads.to_bits(keys, dtype)
    out = to_bits(GpuBatch(wl).decode())
    assert device_error() == 0
    assert every_sequence_error(wl, out) <= TOL[dtype]
    v = formats.decode_bits(wl.values, dtype)
    o = formats.decode_bits(out, dtype)
    for (s, kvh), row in picks.items():  # the selected head returns (about) that V row
        assert np.max(np.abs(o[s, kvh * g] - v[row, kvh])) <= TOL[dtype]


@pytest.mark.parametrize("dtype,hq,hkv", SHAPES)
@pytest.mark.parametrize("k_std", [6.0, 8.0])
def test_wide_score_range(dtype, hq, hkv, k_std):
    """K ~ N(0, std^2): scores with a standard deviation of 6-8 units."""
    wl = batch(dtype, hq, hkv, seed=10 + SHAPES.index((dtype, hq, hkv)), k_std=k_std)
    out = to_bits(GpuBatch(wl).decode())
    assert device_error() == 0
    assert every_sequence_error(wl, out) <= TOL[dtype]


def rising_keys(wl, rise, rng):
    """Add to every key a multiple of its sequence's query direction u (the mean of the
    group's query rows, normalised) that grows linearly along the context, so that the
    score of a head whose query points along u rises by about `rise` units end to end."""
    dtype = wl.dtype
    g = wl.num_q_heads // wl.num_kv_heads
    keys = as_float(wl.keys, dtype)
    q = as_float(wl.q, dtype).astype(np.float64)
    for s in range(wl.num_seqs):
        a, c = int(wl.seq_start[s]), int(wl.context_lens[s])
        for kvh in range(wl.num_kv_heads):
            u = q[s, kvh * g:(kvh + 1) * g].mean(axis=0)
            u /= np.linalg.norm(u)
            qu = float(q[s, kvh * g] @ u)
            slope = rise / max(1, c - 1) / (wl.scale * abs(qu))
            keys[a:a + c, kvh] += (np.sign(qu) * slope * np.arange(c))[:, None] * u[None, :]
    wl.keys = workloads.to_bits(keys, dtype)


@pytest.mark.parametrize("dtype,hq,hkv", SHAPES)
def test_scores_rising_along_the_context(dtype, hq, hkv):
    """The running maximum grows at every stage, and the later pieces of a cut pair hold
    the larger maxima."""
    wl = batch(dtype, hq, hkv, seed=20 + SHAPES.index((dtype, hq, hkv)))
    rising_keys(wl, 60.0, np.random.default_rng(3))
    gb = GpuBatch(wl)
    out = to_bits(gb.decode())
    assert device_error() == 0
    assert every_sequence_error(wl, out) <= TOL[dtype]


def test_fp8_blocks_wide_score_range():
    """FP8 blocks over keys with a spread of 7 (scale = the largest |K| / 448)."""
    from oracle import fp8
    wl = batch("bf16", 32, 8, seed=30, k_std=7.0)
    kmax = float(np.abs(formats.decode_bits(wl.keys, "bf16")).max())
    vmax = float(np.abs(formats.decode_bits(wl.values, "bf16")).max())
    ks, vs = kmax / 448.0, vmax / 448.0
    from test_gpu_fp8 import Fp8Batch, oracle_place as fp8_place
    gb = Fp8Batch(wl, ks, vs)
    got = gb.decode()
    assert device_error() == 0
    k8, v8, tables = fp8_place(wl, ks, vs)
    ref, err = fp8.paged_decode_bits(wl.q, k8, v8, tables, wl.context_lens, wl.scale, ks, vs,
                                     wl.block_size, wl.dtype)
    assert not err.any()
    assert max_err(got, ref, "bf16") <= TOL["bf16"]


def test_prefill_row_maximum_grows_past_the_rescale_threshold():
    """Causal prefill over scores that rise by about 0.15 per token: a row's running
    maximum grows by far more than 8 (exp2 units) from one 64-key tile to the next, so the
    kernel's lazy rescale of O runs at every tile.  Checked on the inputs themselves
    before the comparison."""
    rng = np.random.default_rng(90)
    ctx, qlen = [700, 2048, 1300], [700, 2048, 260]
    T = max(ctx) // 16 + 1
    wl = workloads._prefill("prefill_peaked", rng, ctx, qlen, "bf16", 32, 8, 128, 16,
                            sum(-(-c // 16) for c in ctx) + 9, T * 16, 1.0 / math.sqrt(128))
    g = 4
    keys = as_float(wl.keys, "bf16")
    q = as_float(wl.q, "bf16")
    u = rng.standard_normal(128)
    u /= np.linalg.norm(u)
    gamma = 4.0                                   # every query row gains gamma * u
    per_token = 0.15 / (wl.scale * gamma)         # key growth along u per position
    for s in range(wl.num_seqs):
        a, c = int(wl.seq_start[s]), int(wl.context_lens[s])
        keys[a:a + c] += (per_token * np.arange(c))[:, None, None] * u[None, None, :]
        qa, qb = int(wl.query_start[s]), int(wl.query_start[s + 1])
        q[qa:qb] += gamma * u[None, None, :]
    wl.keys = workloads.to_bits(keys, "bf16")
    wl.q = workloads.to_bits(q, "bf16")
    # by construction: the scores of the last query row of sequence 1, head 0, per tile
    s = 1
    a, c = int(wl.seq_start[s]), int(wl.context_lens[s])
    kk = formats.decode_bits(wl.keys[a:a + c, 0], "bf16")
    qq = formats.decode_bits(wl.q[int(wl.query_start[s + 1]) - 1, 0], "bf16")
    z = wl.scale * (kk @ qq) * math.log2(math.e)
    tile_max = np.maximum.accumulate([z[i:i + 64].max() for i in range(0, c, 64)])
    assert np.max(np.diff(tile_max)) > 8.0
    gb = GpuBatch(wl)
    qs = torch.from_numpy(wl.query_start.astype(np.int32)).cuda()
    out = pa.prefill(gb.q, gb.k_cache, gb.v_cache, gb.tables, gb.ctx, qs, wl.scale, max(qlen))
    got = to_bits(out)
    assert device_error() == 0
    kc, vc, tables = oracle_place(wl)
    ref, err = oracle_prefill.paged_prefill_bits(wl.q, kc, vc, tables, wl.context_lens,
                                                 wl.query_start, wl.scale, wl.block_size, "bf16")
    assert not err.any()
    assert max_err(got, ref, "bf16") <= TOL["bf16"]
