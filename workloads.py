"""Seeded synthetic inputs shaped like the pages' decode workloads.

This module is the only code shared by the oracle side and the CUDA side of the tests
and the benchmark.  It draws random numbers and nothing else: it holds none of the
method's arithmetic (no address translation, no slots, no attention).  Each side builds
its block tables with its own allocator from ``free_order``, writes the logical K/V rows
with its own cache write, and computes its own attention.

Values are 16-bit floats kept as raw ``uint16`` patterns: float32 normals rounded to
nearest-even by NumPy (fp16) or torch (bf16).  Every recipe uses
``numpy.random.default_rng(seed)`` with seed 0 by default.

Recipes (the shapes of the pages' workloads; no dataset or weights are involved):
    tiny         4 seqs, ctx {7,16,33,100}, B=16, pool 64, 4 q / 2 kv heads, d=64, fp16,
                 q/K/V ~ N(0,1), scale 1/8
    llama31_8b   64 seqs, 32 q / 8 kv heads, d=128, bf16, B=16, ctx ~ U[128, 2048],
                 K/V ~ N(0,1), pool 16384 blocks in shuffled order, plus a cache write of
                 each sequence's newest token
    llama7b_mha  256 seqs, 32 heads (MHA), d=128, fp16, B=16, ctx = clip(round(lognormal(
                 ln 384, 1.0)), 16, 4096) standing in for chat-trace lengths, K/V ~ N(0, 0.5^2),
                 pool 1.25x the blocks the batch needs, shuffled
    beam         2 prompts x 8 beams, 1024-token prefix + 1 shared generated token, then
                 1..15 private tokens per beam; 32 q / 8 kv heads, d=128, bf16, B=16
    long         8 seqs, ctx {8192,16384,24576,32768 x5}, 32 q / 8 kv heads, d=128, bf16,
                 B in {8,16,32}, K/V ~ N(0,1), pool 1.25x the blocks needed, shuffled

Prefill recipes (q holds every new token of every sequence; query_start marks them):
    prefill_tiny        4 seqs, ctx {5,40,100,33}, new tokens {5,17,33,1}, B=16, pool 64,
                        4 q / 2 kv heads, d=64, fp16
    prefill_llama31_8b  8 prompts of 2048 tokens from scratch, 32 q / 8 kv heads, d=128,
                        bf16, B=16, pool 3.3x the blocks one batch needs (three batches
                        rotate in disjoint blocks), shuffled
    prefill_chunked     16 seqs, ctx ~ U[1024, 4096], the last 512 tokens new (a chunk of
                        a longer prompt), otherwise as prefill_llama31_8b

Shared-prefix prompts (prefix caching): every request starts with the same system
prompt; the K/V rows of those positions are the same draw for every request (a model
computes a position's K/V from the tokens up to it), the rest are drawn per request.
Token ids are uniform over a 128256-entry vocabulary.
    prefix_tiny         4 requests, system prompt 40 tokens, own tokens {5,17,33,1}, B=16,
                        4 q / 2 kv heads, d=64, fp16
    prefix_llama31_8b   16 requests, system prompt 1024 tokens, 512 own tokens each,
                        32 q / 8 kv heads, d=128, bf16, B=16
"""
from dataclasses import dataclass, field
import math

import numpy as np


def to_bits(x32, dtype):
    """Round float32 values to fp16/bf16 (nearest-even) and return the uint16 patterns."""
    x32 = np.ascontiguousarray(x32, dtype=np.float32)
    if dtype == "fp16":
        return x32.astype(np.float16).view(np.uint16)
    if dtype == "bf16":
        import torch
        t = torch.from_numpy(x32).to(torch.bfloat16)
        return t.view(torch.int16).numpy().view(np.uint16)
    raise ValueError(dtype)


def normal_bits(rng, shape, std, dtype):
    return to_bits(rng.standard_normal(shape, dtype=np.float32) * np.float32(std), dtype)


@dataclass
class DecodeWorkload:
    """One decode batch: logical K/V rows per sequence plus a pool to place them in."""
    name: str
    dtype: str                  # "fp16" | "bf16"
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int             # physical blocks in the pool
    max_blocks_per_seq: int     # width T of the block table
    scale: float
    context_lens: np.ndarray    # int32 [n]
    free_order: np.ndarray      # int32 [num_blocks]: initial free-list order (seeded shuffle)
    q: np.ndarray               # uint16 [n, Hq, d]
    keys: np.ndarray            # uint16 [sum(ctx), Hkv, d]: logical rows, one sequence after another
    values: np.ndarray          # uint16 [sum(ctx), Hkv, d]
    seq_start: np.ndarray       # int64 [n + 1]: rows of sequence s are keys[seq_start[s]:seq_start[s+1]]
    notes: dict = field(default_factory=dict)

    @property
    def num_seqs(self):
        return len(self.context_lens)


def _decode(name, rng, ctx, dtype, hq, hkv, d, bsz, num_blocks, max_ctx, scale, kv_std,
            q_std=1.0, notes=None):
    ctx = np.asarray(ctx, dtype=np.int32)
    total = int(ctx.sum())
    q = normal_bits(rng, (len(ctx), hq, d), q_std, dtype)
    keys = normal_bits(rng, (total, hkv, d), kv_std, dtype)
    values = normal_bits(rng, (total, hkv, d), kv_std, dtype)
    seq_start = np.zeros(len(ctx) + 1, dtype=np.int64)
    np.cumsum(ctx, out=seq_start[1:])
    free_order = rng.permutation(num_blocks).astype(np.int32)
    return DecodeWorkload(name=name, dtype=dtype, num_q_heads=hq, num_kv_heads=hkv,
                          head_dim=d, block_size=bsz, num_blocks=num_blocks,
                          max_blocks_per_seq=max_ctx // bsz, scale=scale, context_lens=ctx,
                          free_order=free_order, q=q, keys=keys, values=values,
                          seq_start=seq_start, notes=dict(notes or {}))


def _pool_for(ctx, bsz, slack=1.25):
    """Pool size for 'random placement' recipes that name no pool: 1.25x the blocks needed."""
    return int(math.ceil(slack * sum(-(-int(c) // bsz) for c in ctx)))


def tiny(seed=0):
    rng = np.random.default_rng(seed)
    return _decode("tiny", rng, [7, 16, 33, 100], "fp16", 4, 2, 64, 16, 64, 128,
                   1.0 / math.sqrt(64), 1.0)


def llama31_8b(seed=0, num_seqs=64):
    rng = np.random.default_rng(seed)
    ctx = rng.integers(128, 2048, size=num_seqs, endpoint=True)
    return _decode("llama31_8b", rng, ctx, "bf16", 32, 8, 128, 16, 16384, 2048,
                   1.0 / math.sqrt(128), 1.0, notes={"new_token_per_seq": True})


def llama7b_mha(seed=0, num_seqs=256):
    rng = np.random.default_rng(seed)
    ctx = np.clip(np.rint(rng.lognormal(math.log(384.0), 1.0, size=num_seqs)), 16, 4096)
    ctx = ctx.astype(np.int32)
    return _decode("llama7b_mha", rng, ctx, "fp16", 32, 32, 128, 16, _pool_for(ctx, 16), 4096,
                   1.0 / math.sqrt(128), 0.5)


def long_context(block_size=16, seed=0):
    rng = np.random.default_rng(seed)
    ctx = [8192, 16384, 24576] + [32768] * 5
    return _decode(f"long_b{block_size}", rng, ctx, "bf16", 32, 8, 128, block_size,
                   _pool_for(ctx, block_size), 32768, 1.0 / math.sqrt(128), 1.0)


def custom(name, context_lens, dtype, num_q_heads, num_kv_heads, head_dim, block_size,
           num_blocks, max_context, scale=None, kv_std=1.0, seed=0):
    """A decode batch of any shape (tests use it for edge cases and ragged tails)."""
    rng = np.random.default_rng(seed)
    scale = 1.0 / math.sqrt(head_dim) if scale is None else scale
    return _decode(name, rng, context_lens, dtype, num_q_heads, num_kv_heads, head_dim,
                   block_size, num_blocks, max_context, scale, kv_std)


@dataclass
class BeamWorkload:
    """Shared-prefix beams: each prompt holds ``prefix_tokens`` prompt tokens plus one
    generated token before it forks into ``beams`` beams; beam b then generates
    ``private_tokens[b]`` tokens of its own."""
    dtype: str
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    max_blocks_per_seq: int
    scale: float
    prompts: int
    beams: int
    shared_tokens: int          # tokens each prompt holds before the fork (1024 + 1)
    private_tokens: np.ndarray  # int32 [prompts * beams], each in 1..15
    free_order: np.ndarray      # int32 [num_blocks]
    shared_keys: np.ndarray     # uint16 [prompts, shared_tokens, Hkv, d]
    shared_values: np.ndarray
    private_keys: list          # per beam: uint16 [private_tokens[b], Hkv, d]
    private_values: list
    q: np.ndarray               # uint16 [prompts * beams, Hq, d]


def beam(seed=0, prompts=2, beams=8, prefix=1024, num_blocks=256):
    rng = np.random.default_rng(seed)
    dtype, hq, hkv, d, bsz = "bf16", 32, 8, 128, 16
    shared = prefix + 1
    priv = rng.integers(1, 15, size=prompts * beams, endpoint=True).astype(np.int32)
    shared_k = normal_bits(rng, (prompts, shared, hkv, d), 1.0, dtype)
    shared_v = normal_bits(rng, (prompts, shared, hkv, d), 1.0, dtype)
    pk = [normal_bits(rng, (int(t), hkv, d), 1.0, dtype) for t in priv]
    pv = [normal_bits(rng, (int(t), hkv, d), 1.0, dtype) for t in priv]
    q = normal_bits(rng, (prompts * beams, hq, d), 1.0, dtype)
    free_order = rng.permutation(num_blocks).astype(np.int32)
    return BeamWorkload(dtype=dtype, num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                        block_size=bsz, num_blocks=num_blocks, max_blocks_per_seq=72,
                        scale=1.0 / math.sqrt(d), prompts=prompts, beams=beams,
                        shared_tokens=shared, private_tokens=priv, free_order=free_order,
                        shared_keys=shared_k, shared_values=shared_v, private_keys=pk,
                        private_values=pv, q=q)


@dataclass
class PrefillWorkload(DecodeWorkload):
    """A prefill batch: like a decode batch, but q holds the newest q_len_s tokens of every
    sequence, rows query_start[s] .. query_start[s+1]-1 (q is [total new tokens, Hq, d])."""
    query_start: np.ndarray = None  # int64 [n + 1]


def _prefill(name, rng, ctx, qlen, dtype, hq, hkv, d, bsz, num_blocks, max_ctx, scale,
             kv_std=1.0, q_std=1.0):
    base = _decode(name, rng, ctx, dtype, hq, hkv, d, bsz, num_blocks, max_ctx, scale, kv_std)
    qlen = np.asarray(qlen, dtype=np.int64)
    query_start = np.zeros(len(qlen) + 1, dtype=np.int64)
    np.cumsum(qlen, out=query_start[1:])
    q = normal_bits(rng, (int(query_start[-1]), hq, d), q_std, dtype)
    fields = {k: getattr(base, k) for k in base.__dataclass_fields__}
    fields["q"] = q
    return PrefillWorkload(**fields, query_start=query_start)


def prefill_tiny(seed=0):
    rng = np.random.default_rng(seed)
    return _prefill("prefill_tiny", rng, [5, 40, 100, 33], [5, 17, 33, 1], "fp16", 4, 2, 64,
                    16, 64, 128, 1.0 / math.sqrt(64))


def prefill_llama31_8b(seed=0, num_seqs=8, prompt=2048):
    rng = np.random.default_rng(seed)
    ctx = [prompt] * num_seqs
    return _prefill("prefill_llama31_8b", rng, ctx, ctx, "bf16", 32, 8, 128, 16,
                    int(3.3 * num_seqs * (prompt // 16)), prompt, 1.0 / math.sqrt(128))


def prefill_chunked(seed=0, num_seqs=16, chunk=512):
    rng = np.random.default_rng(seed)
    ctx = rng.integers(1024, 4096, size=num_seqs, endpoint=True)
    return _prefill("prefill_chunked", rng, ctx, [chunk] * num_seqs, "bf16", 32, 8, 128, 16,
                    int(3.3 * sum(-(-int(c) // 16) for c in ctx)), 4096, 1.0 / math.sqrt(128))


@dataclass
class PrefixWorkload(PrefillWorkload):
    """Prompts from scratch that share a system prompt: q holds every token of every
    prompt; tokens holds their ids (int32 [sum(ctx)], same layout as keys)."""
    tokens: np.ndarray = None
    system_len: int = 0


def _prefix(name, rng, system_len, own, dtype, hq, hkv, d, bsz, num_blocks, scale,
            vocab=128256):
    own = np.asarray(own, dtype=np.int32)
    ctx = system_len + own
    base = _prefill(name, rng, ctx, ctx, dtype, hq, hkv, d, bsz, num_blocks,
                    int(-(-int(ctx.max()) // bsz) * bsz), scale)
    sys_tok = rng.integers(0, vocab, size=system_len).astype(np.int32)
    sys_k = normal_bits(rng, (system_len, hkv, d), 1.0, dtype)
    sys_v = normal_bits(rng, (system_len, hkv, d), 1.0, dtype)
    toks = []
    for s in range(len(ctx)):
        a = int(base.seq_start[s])
        base.keys[a:a + system_len] = sys_k
        base.values[a:a + system_len] = sys_v
        toks.append(np.concatenate([sys_tok, rng.integers(0, vocab, size=int(own[s])).astype(np.int32)]))
    fields = {k: getattr(base, k) for k in base.__dataclass_fields__}
    return PrefixWorkload(**fields, tokens=np.concatenate(toks), system_len=system_len)


def prefix_tiny(seed=0):
    rng = np.random.default_rng(seed)
    return _prefix("prefix_tiny", rng, 40, [5, 17, 33, 1], "fp16", 4, 2, 64, 16, 64,
                   1.0 / math.sqrt(64))


def prefix_llama31_8b(seed=0, num_reqs=16, system_len=1024, own=512):
    rng = np.random.default_rng(seed)
    return _prefix("prefix_llama31_8b", rng, system_len, [own] * num_reqs, "bf16", 32, 8, 128,
                   16, 4 * num_reqs * ((system_len + own) // 16), 1.0 / math.sqrt(128))


RECIPES = {
    "tiny": tiny,
    "llama31_8b": llama31_8b,
    "llama7b_mha": llama7b_mha,
    "long_b8": lambda seed=0: long_context(8, seed),
    "long_b16": lambda seed=0: long_context(16, seed),
    "long_b32": lambda seed=0: long_context(32, seed),
    "beam": beam,
    "prefill_tiny": prefill_tiny,
    "prefill_llama31_8b": prefill_llama31_8b,
    "prefill_chunked": prefill_chunked,
    "prefix_tiny": prefix_tiny,
    "prefix_llama31_8b": prefix_llama31_8b,
}
