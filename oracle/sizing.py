"""Closed forms the pages print (test infrastructure only).

* Blocks for S tokens: N = ceil(S / B) (aiqz.cc "vLLM PagedAttention engine", section
  分页存储设计); the unused slots of the last block, N*B - S, are the only internal waste
  (daiw.org "Paged Attention", section 定义 table; horeb.top, section 分配策略).
* KV bytes of one sequence: 2 * L * s * h_kv * d_h * b (daiw.org, section 回顾与衔接;
  aiqz.cc section KV缓存之谜 writes it M_KV = 2 x L x H x d x S x b x P with batch b and
  element bytes P).
* Bytes of one block: 2 * L * B * h_kv * d_h * b (daiw.org, section 工程现场, step 2).
* Capacity: blocks = pool bytes // bytes per block; concurrency = blocks // blocks per
  sequence (daiw.org, section 工程现场, steps 3-5).
* Fragmentation eta = 1 - sum S_i / sum S_i^max (aiqz.cc, section 连续分配之殇) and
  effective utilisation U = sum S_used / sum S_alloc (aiqz.cc, section 新旧方案对比).
"""
import math


def blocks_needed(tokens, block_size):
    return math.ceil(tokens / block_size)


def tail_waste(tokens, block_size):
    return blocks_needed(tokens, block_size) * block_size - tokens


def kv_bytes_per_sequence(layers, tokens, kv_heads, head_dim, elem_bytes, batch=1):
    return 2 * layers * kv_heads * head_dim * tokens * batch * elem_bytes


def kv_bytes_per_block(layers, block_size, kv_heads, head_dim, elem_bytes):
    return 2 * layers * block_size * kv_heads * head_dim * elem_bytes


def pool_blocks(pool_bytes, block_bytes):
    return pool_bytes // block_bytes


def max_concurrency(num_blocks, tokens_per_seq, block_size):
    return num_blocks // blocks_needed(tokens_per_seq, block_size)


def fragmentation(used_tokens, reserved_tokens):
    return 1.0 - sum(used_tokens) / sum(reserved_tokens)


def effective_utilisation(used_tokens, allocated_tokens):
    return sum(used_tokens) / sum(allocated_tokens)
