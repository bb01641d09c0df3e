"""GPU parity of prefix-cached prefill: requests that share a system prompt are placed
through the C++ pool's prefix cache (the second and later requests reuse the system
prompt's full blocks, write K/V only for the rest and prefill only the rest); the
outputs equal the oracle's prefill of every whole prompt (placed without any cache)
within tolerance, and equal the GPU's own uncached prefill of the whole prompts bit for
bit; the cached-token counts and tables match the oracle pool."""
import numpy as np
import pytest
import torch

import paged_kv_cache_149_gb300 as pa
import workloads
from gpu_harness import TOL, device_error, max_err, nan_cache, oracle_place, to_bits, to_device
from oracle import prefill as oracle_prefill
from oracle.block_pool import BlockPool as OraclePool

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(libpa):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    device_error()


def place(wl, use_cache):
    """Requests one after another through the library pool; K/V written only for the
    positions not found cached.  Returns caches, tables and per-request cached tokens."""
    n, T = wl.num_seqs, wl.max_blocks_per_seq
    pool = pa.BlockPool(wl.num_blocks, wl.block_size, wl.free_order)
    kc = nan_cache(wl.num_blocks, wl.num_kv_heads, wl.block_size, wl.head_dim, wl.dtype)
    vc = nan_cache(wl.num_blocks, wl.num_kv_heads, wl.block_size, wl.head_dim, wl.dtype)
    keys, values = to_device(wl.keys, wl.dtype), to_device(wl.values, wl.dtype)
    tables = np.full((n, T), -1, dtype=np.int32)
    cached = []
    for s in range(n):
        a, b = int(wl.seq_start[s]), int(wl.seq_start[s + 1])
        if use_cache:
            c = pool.allocate_prefix(s, wl.tokens[a:b])
        else:
            pool.allocate(s, b - a)
            c = 0
        cached.append(c)
        if b - a - c > 0:
            slots = torch.from_numpy(pool.slots(s, c, b - a - c)).cuda()
            pa.reshape_and_cache(keys[a + c:b], values[a + c:b], kc, vc, slots)
        t = pool.block_table(s)
        tables[s, :len(t)] = t
    return kc, vc, tables, np.array(cached)


def prefill_rows(wl, kc, vc, tables, cached):
    """Prefill of each request's uncached tokens (over its whole context)."""
    q = to_device(wl.q, wl.dtype)
    rows = np.concatenate([np.arange(wl.query_start[s] + cached[s], wl.query_start[s + 1])
                           for s in range(wl.num_seqs)])
    own = wl.context_lens - cached
    qs = np.zeros(wl.num_seqs + 1, dtype=np.int32)
    np.cumsum(own, out=qs[1:])
    out = pa.prefill(q[torch.from_numpy(rows).cuda()].contiguous(), kc, vc,
                     torch.from_numpy(tables).cuda(),
                     torch.from_numpy(wl.context_lens.astype(np.int32)).cuda(),
                     torch.from_numpy(qs).cuda(), wl.scale, int(own.max()))
    torch.cuda.synchronize()
    return rows, to_bits(out)


@pytest.mark.parametrize("recipe,check_seqs", [("prefix_tiny", None),
                                               ("prefix_llama31_8b", [1, 15])])
def test_cached_prefill_matches_the_oracle(recipe, check_seqs):
    wl = workloads.RECIPES[recipe]()
    kc, vc, tables, cached = place(wl, True)
    assert device_error() == 0
    # bookkeeping: the oracle pool finds the same hits and builds the same tables
    ref = OraclePool(wl.num_blocks, wl.block_size, wl.free_order)
    for s in range(wl.num_seqs):
        a, b = int(wl.seq_start[s]), int(wl.seq_start[s + 1])
        assert ref.allocate_prefix(s, wl.tokens[a:b]) == cached[s]
        assert ref.block_table(s) == list(tables[s][:len(ref.block_table(s))])
    full = (wl.system_len // wl.block_size) * wl.block_size
    assert cached[0] == 0 and all(c == full for c in cached[1:])
    rows, got = prefill_rows(wl, kc, vc, tables, cached)
    assert device_error() == 0
    okc, ovc, otables = oracle_place(wl)
    want, err = oracle_prefill.paged_prefill_bits(wl.q, okc, ovc, otables, wl.context_lens,
                                                  wl.query_start, wl.scale, wl.block_size,
                                                  wl.dtype, seqs=check_seqs)
    assert not err.any()
    seqs = range(wl.num_seqs) if check_seqs is None else check_seqs
    pos = {r: i for i, r in enumerate(rows)}
    for s in seqs:
        rr = np.arange(wl.query_start[s] + cached[s], wl.query_start[s + 1])
        e = max_err(got[[pos[r] for r in rr]], want[rr], wl.dtype)
        assert e <= TOL[wl.dtype], (s, e)


@pytest.mark.parametrize("recipe", ["prefix_tiny", "prefix_llama31_8b"])
def test_cached_prefill_is_bit_identical_to_uncached(recipe):
    wl = workloads.RECIPES[recipe]()
    kc, vc, tables, cached = place(wl, True)
    rows, got = prefill_rows(wl, kc, vc, tables, cached)
    kc0, vc0, tables0, zero = place(wl, False)
    rows0, full = prefill_rows(wl, kc0, vc0, tables0, zero)
    assert device_error() == 0
    np.testing.assert_array_equal(got, full[rows])
