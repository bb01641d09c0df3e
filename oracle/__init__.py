"""Plain CPU oracle for paged decode attention.

TEST INFRASTRUCTURE ONLY.  Nothing in the product package imports this package, and it
imports nothing from the product package: the two share no code.  Only ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py`` (its ``cpu_baseline`` leg and its
``--impl reference`` arm) may import or run it.

Everything here is float64 NumPy (or pure Python on tiny cases) written for a reader
to check by eye against the pages it follows:

* daiw.org, "Paged Attention" (从 Bit 到 AGI, chapter 8) -- sections 直觉, 定义, 例子,
  量化, 工程现场, 动手试一试, 回顾与衔接, 速查卡.
* chenyuan1125.github.io, "vllm-pagedattention" -- sections "页表真正解开的，是逻辑连续和
  物理连续", "一块内存，如何安全地属于多条序列", "它和 FlashAttention 优化的是两张不同的账".
* aiqz.cc, "vLLM PagedAttention engine" -- sections KV缓存之谜, 连续分配之殇,
  分页存储设计, 新旧方案对比, Python 演示.
* horeb.top, "vLLM PagedAttention：大模型推理的显存管理革命" -- sections 背景,
  "PagedAttention：从操作系统借来的分页" (分配策略), "内存共享：写时复制".

Modules:
    formats     -- 16-bit float encodings and round-to-nearest-even from float64.
    attention   -- paged decode attention, its split-KV partials and their merge.
    cache_ops   -- reshape_and_cache (slot writes), copy_blocks and swap_blocks (block
                   copies within a pool and between the device and a CPU pool).
    block_pool  -- free list, reference counts, fork, copy-on-write and swap bookkeeping.
    sizing      -- the closed forms the pages print (block counts, bytes, capacity).
    prefill     -- causal multi-query attention of each sequence's newest tokens.
    fp8         -- FP8 (E4M3) KV blocks: the format, the quantising cache write, decode.
    int4        -- INT4 KV blocks (codes with one scale per row): the format, the
                   quantising cache write, decode.

Every function is pinned by ``tests/test_oracle_*.py`` against something other than
itself: values the pages print, closed forms, library special cases (NumPy float16,
torch scaled_dot_product_attention in float64) and brute force on tiny inputs.
"""
