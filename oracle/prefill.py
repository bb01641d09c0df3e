"""Paged prefill (multi-query, causal) attention as its plain definition (test
infrastructure only).

What it computes.  A prompt, or a chunk of one, is processed before decoding starts: its
blocks are allotted first, ceil(prompt_tokens / 16) of them (horeb.top "vLLM
PagedAttention：大模型推理的显存管理革命", section 分配策略); prefill handles large blocks of
queries while decode handles one (chenyuan1125 "vllm-pagedattention", section 它和
FlashAttention…), and a kernel has to read the block table to combine FlashAttention's
tiling with paging (daiw.org "Paged Attention", section 回顾与衔接).  Paging changes only
where rows live, so the oracle is ordinary causal attention over each sequence's logical
rows:

    sequence s owns query rows query_start[s] .. query_start[s+1]-1: its newest
    q_len_s = query_start[s+1] - query_start[s] tokens, at positions
    p = ctx_s - q_len_s .. ctx_s - 1 of its context (their K/V rows are already in the
    cache, like every earlier token's);
    the token at position p attends to positions 0 .. p:
        z_t = scale * <q[row, h], K_s[t, h // G]>,  t <= p
        out[row, h] = sum_t softmax(z)_t V_s[t, h // G]

The rows are gathered one token at a time through the table (attention.logical_rows);
scores, max-subtracted softmax and the weighted sum are float64, rounded once at the end.
"""
import numpy as np

from .attention import ERR_BAD_CONTEXT, logical_rows, validate_item
from .formats import decode_bits, encode_bits


def paged_prefill(q_bits, k_cache_bits, v_cache_bits, block_tables, context_lens,
                  query_start, scale, block_size, dtype, seqs=None):
    """Returns (out float64 [num_q_rows, Hq, d], error bits int64 [n]).  A sequence with an
    invalid context, a bad block id among the blocks it uses, or q_len > ctx yields zeros
    and its error bits.  With ``seqs``, only those sequences are computed (the rows of the
    others stay zero)."""
    q_bits = np.asarray(q_bits)
    ntok, hq, d = q_bits.shape
    hkv = k_cache_bits.shape[1]
    g = hq // hkv
    nb = k_cache_bits.shape[0]
    n = len(context_lens)
    out = np.zeros((ntok, hq, d), dtype=np.float64)
    errs = np.zeros(n, dtype=np.int64)
    for s in (range(n) if seqs is None else seqs):
        qs, qe = int(query_start[s]), int(query_start[s + 1])
        qlen, ctx = qe - qs, int(context_lens[s])
        if qlen == 0:
            continue
        err = validate_item(block_tables[s], ctx, block_size, nb)
        if not err and qlen > ctx:
            err = ERR_BAD_CONTEXT
        errs[s] = err
        if err:
            continue
        k = logical_rows(k_cache_bits, block_tables[s], ctx, block_size, dtype)
        v = logical_rows(v_cache_bits, block_tables[s], ctx, block_size, dtype)
        q = decode_bits(q_bits[qs:qe], dtype)                     # [qlen, Hq, d]
        pos = ctx - qlen + np.arange(qlen)                         # position of each query
        future = np.arange(ctx)[None, :] > pos[:, None]            # keys after the query
        for h in range(hq):
            z = scale * (q[:, h, :] @ k[:, h // g, :].T)           # [qlen, ctx]
            z[future] = -np.inf
            z = z - z.max(axis=1, keepdims=True)
            w = np.exp(z)
            w = w / w.sum(axis=1, keepdims=True)
            out[qs:qe, h, :] = w @ v[:, h // g, :]
    return out, errs


def paged_prefill_bits(*args, **kw):
    """paged_prefill rounded to the 16-bit output format (RNE); also the error bits."""
    dtype = args[8] if len(args) > 8 else kw["dtype"]
    out, err = paged_prefill(*args, **kw)
    return encode_bits(out, dtype), err
