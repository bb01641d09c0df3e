"""Cache writes and block copies, element by element (test infrastructure only).

reshape_and_cache: a new token's K/V row goes into the free slot of its sequence's last
block, and a fresh block is appended to the table when the last one is full
(chenyuan1125 "vllm-pagedattention", section 页表真正解开的…; horeb.top, section 分配策略).
The slot number of token t is ``block_table[t // B] * B + t % B``; the row is written at
block ``slot // B``, row ``slot % B``.  A negative slot means "no write".

copy_blocks: when a branch must write into a last block that is still shared, that
block is copied, the branch's mapping is updated, then the write goes ahead; full old
blocks stay shared (chenyuan1125, section 一块内存，如何安全地属于多条序列; horeb.top,
section 内存共享：写时复制).  A copy moves every kv head and every row of the block.

swap_blocks: a preempted request's blocks move whole between the device pool and a
CPU pool, and back when room returns (aiqz.cc "vLLM PagedAttention engine", section
连续批处理：随到随走的新秩序): block dst of the destination pool := block src of the source
pool, every kv head and row.

All are exact copies of 16-bit patterns; the oracle works on ``uint16`` arrays.
"""
import numpy as np


def slot_of(table_row, t, block_size):
    """Slot number of logical token t: physical block * B + row within the block."""
    return int(table_row[t // block_size]) * block_size + t % block_size


def reshape_and_cache(k_cache, v_cache, key, value, slot_mapping):
    """Return copies of (k_cache, v_cache) with row i of key/value written at its slot.

    k_cache, v_cache [NB, Hkv, B, d] uint16; key, value [n_tok, Hkv, d] uint16;
    slot_mapping [n_tok] int64.  Slots < 0 are skipped; a slot >= NB*B raises (the device
    path skips it and flags it).  Two tokens naming the same slot are rejected: the
    write order would be undefined.
    """
    nb, hkv, b, d = k_cache.shape
    k_out = k_cache.copy()
    v_out = v_cache.copy()
    seen = set()
    for i, slot in enumerate(np.asarray(slot_mapping, dtype=np.int64)):
        slot = int(slot)
        if slot < 0:
            continue
        if slot >= nb * b:
            raise IndexError(f"slot {slot} outside the pool of {nb * b} slots")
        if slot in seen:
            raise ValueError(f"slot {slot} written twice in one call")
        seen.add(slot)
        blk, row = slot // b, slot % b
        k_out[blk, :, row, :] = key[i]
        v_out[blk, :, row, :] = value[i]
    return k_out, v_out


def copy_blocks(k_cache, v_cache, pairs):
    """Return copies of the caches with block dst := block src for every (src, dst) pair.

    Pairs must not alias: every dst is distinct, and no dst is also a src (so the result
    does not depend on the order of the pairs).  Ids must lie in [0, NB).
    """
    nb = k_cache.shape[0]
    pairs = [(int(s), int(d)) for s, d in np.asarray(pairs, dtype=np.int64).reshape(-1, 2)]
    dsts = [d for _, d in pairs]
    if len(set(dsts)) != len(dsts) or set(dsts) & {s for s, _ in pairs}:
        raise ValueError("copy_blocks pairs alias")
    for s, d in pairs:
        if not (0 <= s < nb and 0 <= d < nb):
            raise IndexError(f"block pair ({s}, {d}) outside [0, {nb})")
    k_out = k_cache.copy()
    v_out = v_cache.copy()
    for s, d in pairs:
        k_out[d] = k_cache[s]
        v_out[d] = v_cache[s]
    return k_out, v_out


def swap_blocks(src_k, src_v, dst_k, dst_v, pairs):
    """Return copies of (dst_k, dst_v) with dst[d] := src[s] for every (s, d) pair.

    The source and destination are different pools (shapes [NBs, Hkv, B, d] and
    [NBd, Hkv, B, d]); destination ids must be distinct; ids must lie in their pool.
    """
    nbs, nbd = src_k.shape[0], dst_k.shape[0]
    pairs = [(int(s), int(d)) for s, d in np.asarray(pairs, dtype=np.int64).reshape(-1, 2)]
    dsts = [d for _, d in pairs]
    if len(set(dsts)) != len(dsts):
        raise ValueError("swap_blocks destinations repeat")
    for s, d in pairs:
        if not (0 <= s < nbs and 0 <= d < nbd):
            raise IndexError(f"block pair ({s}, {d}) outside [0, {nbs}) x [0, {nbd})")
    k_out = dst_k.copy()
    v_out = dst_v.copy()
    for s, d in pairs:
        k_out[d] = src_k[s]
        v_out[d] = src_v[s]
    return k_out, v_out
