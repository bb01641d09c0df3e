"""Helpers for the GPU parity tests: place a workload through the library (C++ pool,
cache-write kernel) and, independently, through the oracle; compare outputs."""
import numpy as np
import torch

import paged_kv_cache_149_gb300 as pa
from oracle import attention, cache_ops, formats
from oracle.block_pool import BlockPool as OraclePool

# max |gpu - oracle| allowed on decode outputs, by output dtype
TOL = {"fp16": 4e-3, "bf16": 1.6e-2}
TORCH_DTYPE = {"fp16": torch.float16, "bf16": torch.bfloat16}


def to_device(bits, dtype, device="cuda"):
    """uint16 patterns -> a torch tensor of the 16-bit dtype (exact)."""
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.to(device).view(TORCH_DTYPE[dtype])


def to_bits(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def nan_cache(num_blocks, hkv, bs, d, dtype, device="cuda"):
    """A cache whose every slot holds the dtype's quiet NaN, so reads of unwritten
    slots show up in the output."""
    nan = formats.FORMATS[dtype]["qnan"]
    t = torch.full((num_blocks, hkv, bs, d), np.int16(np.uint16(nan).view(np.int16)).item(),
                   dtype=torch.int16, device=device)
    return t.view(TORCH_DTYPE[dtype])


class GpuBatch:
    """The library's side: C++ pool tables, slots from the pool, K/V written by
    pa.reshape_and_cache into NaN-filled caches."""

    def __init__(self, wl, device="cuda", free_order=None, seq_ids=None):
        self.wl = wl
        n, T = wl.num_seqs, wl.max_blocks_per_seq
        order = wl.free_order if free_order is None else free_order
        self.pool = pa.BlockPool(wl.num_blocks, wl.block_size, order)
        self.seq_ids = list(range(n)) if seq_ids is None else list(seq_ids)
        tables = np.full((n, T), -1, dtype=np.int32)
        slots = []
        for i, s in enumerate(self.seq_ids):
            c = int(wl.context_lens[i])
            self.pool.allocate(s, c)
            t = self.pool.block_table(s)
            tables[i, :len(t)] = t
            slots.append(self.pool.slots(s, 0, c))
        self.tables_np = tables
        self.k_cache = nan_cache(wl.num_blocks, wl.num_kv_heads, wl.block_size, wl.head_dim, wl.dtype, device)
        self.v_cache = nan_cache(wl.num_blocks, wl.num_kv_heads, wl.block_size, wl.head_dim, wl.dtype, device)
        slot_t = torch.from_numpy(np.concatenate(slots) if slots else np.zeros(0, np.int64)).to(device)
        pa.reshape_and_cache(to_device(wl.keys, wl.dtype, device), to_device(wl.values, wl.dtype, device),
                             self.k_cache, self.v_cache, slot_t)
        self.q = to_device(wl.q, wl.dtype, device)
        self.tables = torch.from_numpy(tables).to(device)
        self.ctx = torch.from_numpy(np.ascontiguousarray(wl.context_lens, dtype=np.int32)).to(device)
        self.workspace = pa.make_workspace(wl.num_q_heads, wl.num_kv_heads, wl.head_dim, device)

    def decode(self, out=None):
        return pa.decode(self.q, self.k_cache, self.v_cache, self.tables, self.ctx, self.wl.scale,
                         out=out, workspace=self.workspace)


def oracle_place(wl):
    """The oracle's side: its own pool and its own cache write."""
    pool = OraclePool(wl.num_blocks, wl.block_size, wl.free_order)
    tables = np.full((wl.num_seqs, wl.max_blocks_per_seq), -1, dtype=np.int32)
    slots = []
    for s in range(wl.num_seqs):
        c = int(wl.context_lens[s])
        pool.allocate(s, c)
        t = pool.block_table(s)
        tables[s, :len(t)] = t
        slots += [pool.slot(s, i) for i in range(c)]
    nan = formats.FORMATS[wl.dtype]["qnan"]
    shape = (wl.num_blocks, wl.num_kv_heads, wl.block_size, wl.head_dim)
    kc = np.full(shape, nan, dtype=np.uint16)
    vc = np.full(shape, nan, dtype=np.uint16)
    kc, vc = cache_ops.reshape_and_cache(kc, vc, wl.keys, wl.values, np.array(slots, dtype=np.int64))
    return kc, vc, tables


def oracle_rows(wl, s):
    """Logical K/V rows of sequence s straight from the workload (float64)."""
    a, b = wl.seq_start[s], wl.seq_start[s + 1]
    return (formats.decode_bits(wl.keys[a:b], wl.dtype), formats.decode_bits(wl.values[a:b], wl.dtype))


def oracle_seq_bits(wl, s):
    """Oracle output of one sequence from its logical rows, rounded to the dtype (RNE)."""
    k, v = oracle_rows(wl, s)
    o = attention.attend(formats.decode_bits(wl.q[s], wl.dtype), k, v, wl.scale)
    return formats.encode_bits(o, wl.dtype)


def max_err(gpu_bits, ref_bits, dtype):
    g = formats.decode_bits(gpu_bits, dtype)
    r = formats.decode_bits(ref_bits, dtype)
    assert not np.isnan(g).any(), "GPU output holds NaN"
    return float(np.max(np.abs(g - r))) if g.size else 0.0


def device_error():
    return pa.get_device_error()
