"""Paged decode attention, written as its plain definition (test infrastructure only).

What the method computes.  Paging changes where K/V rows live, not the attention itself:
the pages say the attention mathematics is unchanged and only the way cache addresses
are obtained changes (chenyuan1125 "vllm-pagedattention", section 页表真正解开的…), and
that not one byte of the cache is altered (aiqz.cc "vLLM PagedAttention engine", section
新旧方案对比).  So the oracle is ordinary single-query attention over each sequence's
logical K/V rows, where logical token t of sequence s lives in physical block
``block_table[s][t // B]`` (daiw.org "Paged Attention", section 直觉; aiqz.cc section
分页存储设计, N_i = ceil(S_i / B) and BlockTable_i[j]) at row ``t % B`` of that block.

Layout read by the oracle (the layout is the build's choice; the pages fix only the table):
    q            [n, Hq, d]          16-bit patterns
    k/v cache    [NB, Hkv, B, d]     16-bit patterns; one kv head of one block is B*d values
    block_tables [n, T] int32        entry j = physical block of logical block j
    context_lens [n] int32

Query head h reads kv head h // G with G = Hq // Hkv (contiguous groups; the pages only
name GQA as a way to cut KV bytes, daiw.org section 量化 callout).

Scores are z_t = scale * <q_h, K_t>; weights are the softmax of z with the maximum
subtracted; the output is sum_t w_t V_t.  All in float64, rounded once at the end.
"""
import numpy as np

from .formats import decode_bits, encode_bits

# Device error bits the product documents for invalid work items.  The oracle mirrors
# the *result* of that convention (zeros for the item) so tests can compare outputs.
ERR_BAD_BLOCK = 1
ERR_BAD_CONTEXT = 2


def logical_rows(cache_bits, table_row, ctx, block_size, dtype):
    """Gather a sequence's logical rows: row t = cache[table_row[t // B], :, t % B, :].

    Returns float64 [ctx, Hkv, d].  One token at a time, exactly as the address
    translation is stated (daiw.org "Paged Attention", section 直觉).
    """
    nb, hkv, b, d = cache_bits.shape
    assert b == block_size
    out = np.empty((ctx, hkv, d), dtype=np.float64)
    for t in range(ctx):
        blk = int(table_row[t // block_size])
        out[t] = decode_bits(cache_bits[blk, :, t % block_size, :], dtype)
    return out


def attend(q_heads, k_rows, v_rows, scale):
    """Ordinary single-query attention for one sequence, float64.

    q_heads [Hq, d]; k_rows, v_rows [ctx, Hkv, d]; returns [Hq, d].
    """
    hq = q_heads.shape[0]
    hkv = k_rows.shape[1]
    g = hq // hkv
    out = np.empty((hq, q_heads.shape[1]), dtype=np.float64)
    for h in range(hq):
        kvh = h // g
        z = scale * (k_rows[:, kvh, :] @ q_heads[h])
        w = np.exp(z - z.max())
        w = w / w.sum()
        out[h] = w @ v_rows[:, kvh, :]
    return out


def validate_item(table_row, ctx, block_size, num_blocks):
    """Error bits for one sequence under the documented device convention (0 = valid)."""
    t = len(table_row)
    if ctx < 1 or ctx > t * block_size:
        return ERR_BAD_CONTEXT
    nblk = -(-ctx // block_size)
    used = np.asarray(table_row[:nblk], dtype=np.int64)
    if np.any(used < 0) or np.any(used >= num_blocks):
        return ERR_BAD_BLOCK
    return 0


def paged_decode(q_bits, k_cache_bits, v_cache_bits, block_tables, context_lens,
                 scale, block_size, dtype, seqs=None):
    """Paged decode attention for every sequence (or the listed ``seqs``).

    Returns (out float64 [n_sel, Hq, d], error_bits int [n_sel]).  A sequence whose
    context length or used table entries are invalid yields zeros and its error bits,
    matching the library's documented skip-and-flag convention.
    """
    n = q_bits.shape[0]
    seqs = range(n) if seqs is None else seqs
    nb = k_cache_bits.shape[0]
    outs, errs = [], []
    for s in seqs:
        ctx = int(context_lens[s])
        err = validate_item(block_tables[s], ctx, block_size, nb)
        errs.append(err)
        if err:
            outs.append(np.zeros(q_bits.shape[1:], dtype=np.float64))
            continue
        k_rows = logical_rows(k_cache_bits, block_tables[s], ctx, block_size, dtype)
        v_rows = logical_rows(v_cache_bits, block_tables[s], ctx, block_size, dtype)
        outs.append(attend(decode_bits(q_bits[s], dtype), k_rows, v_rows, scale))
    return np.stack(outs), np.array(errs, dtype=np.int64)


def paged_decode_bits(*args, **kw):
    """``paged_decode`` rounded to the 16-bit output format (RNE); also returns error bits."""
    dtype = args[7] if len(args) > 7 else kw["dtype"]
    out, err = paged_decode(*args, **kw)
    return encode_bits(out, dtype), err


# ---------------------------------------------------------------------------------------
# Split-KV: partitions of the logical context and their log-sum-exp merge.
#
# The pages describe scoring, softmax and weighted sum done block by block
# (chenyuan1125, section 页表真正解开的…) and name online softmax as FlashAttention's
# technique (section 它和 FlashAttention…).  Splitting a long context into partitions
# that are reduced afterwards is the same rescaling identity:
#   partition i over logical tokens [i*P, (i+1)*P):
#       m_i = max z,  l_i = sum exp(z - m_i),  acc_i = sum exp(z - m_i) V
#   merge: M = max_i m_i,  L = sum_i l_i exp(m_i - M),  o = sum_i acc_i exp(m_i - M) / L
# ---------------------------------------------------------------------------------------

def partition_partials(z, v, part_tokens):
    """Partials (m [NP], l [NP], acc [NP, d]) of scores z [ctx] and rows v [ctx, d]."""
    ctx = z.shape[0]
    starts = range(0, ctx, part_tokens)
    m = np.empty(len(starts))
    l = np.empty(len(starts))
    acc = np.empty((len(starts), v.shape[1]))
    for i, a in enumerate(starts):
        zz = z[a:a + part_tokens]
        m[i] = zz.max()
        e = np.exp(zz - m[i])
        l[i] = e.sum()
        acc[i] = e @ v[a:a + part_tokens]
    return m, l, acc


def merge_partials(m, l, acc):
    """Log-sum-exp merge of partition partials into the normalised output row."""
    big_m = m.max()
    w = np.exp(m - big_m)
    big_l = (l * w).sum()
    return (acc * w[:, None]).sum(axis=0) / big_l


def split_decode_head(q_row, k_rows_g, v_rows_g, scale, part_tokens):
    """One (sequence, head) through partitions + merge; q_row [d], rows [ctx, d]."""
    z = scale * (k_rows_g @ q_row)
    return merge_partials(*partition_partials(z, v_rows_g, part_tokens))


def contiguous_decode_loops(q_heads, k_rows, v_rows, scale):
    """Brute force with Python floats and loops, for tiny inputs only.

    The same definition as ``attend`` but written element by element, with no NumPy
    reductions, so it can stand as an independent check of the vectorised oracle.
    q_heads [Hq][d], k_rows/v_rows [ctx][Hkv][d] (nested sequences of floats).
    """
    import math
    hq = len(q_heads)
    hkv = len(k_rows[0])
    g = hq // hkv
    d = len(q_heads[0])
    ctx = len(k_rows)
    out = []
    for h in range(hq):
        kvh = h // g
        z = []
        for t in range(ctx):
            acc = 0.0
            for k in range(d):
                acc += q_heads[h][k] * k_rows[t][kvh][k]
            z.append(scale * acc)
        zmax = max(z)
        e = [math.exp(zt - zmax) for zt in z]
        tot = sum(e)
        row = []
        for k in range(d):
            s = 0.0
            for t in range(ctx):
                s += e[t] * v_rows[t][kvh][k]
            row.append(s / tot)
        out.append(row)
    return out
