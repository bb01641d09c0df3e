/*
 * pa.h -- C ABI of libpa.so: paged KV-cache decode attention for GB300 (sm_103a).
 *
 * The KV cache of every sequence is stored in fixed-size physical blocks of
 * block_size (B) tokens.  Logical token t of sequence s lives in physical block
 * block_tables[s][t / B], at row t % B of that block (daiw.org "Paged Attention",
 * section 直觉 and 定义; aiqz.cc "vLLM PagedAttention engine", section 分页存储设计,
 * N_i = ceil(S_i / B) and BlockTable_i[j]).  Attention itself is ordinary softmax
 * attention over the logical sequence; only the way K/V addresses are found changes
 * (chenyuan1125 "vllm-pagedattention", section 页表真正解开的，是逻辑连续和物理连续).
 *
 * Layouts (all row-major, all device memory unless stated otherwise):
 *   q             [num_seqs, num_q_heads, head_dim]              fp16 or bf16
 *   out           [num_seqs, num_q_heads, head_dim]              same dtype as q
 *   k_cache       [num_blocks, num_kv_heads, block_size, head_dim] same dtype
 *   v_cache       [num_blocks, num_kv_heads, block_size, head_dim] same dtype
 *   block_tables  [num_seqs, max_blocks_per_seq] int32; entries past ceil(ctx/B) unread
 *   context_lens  [num_seqs] int32, the number of tokens each query attends to
 *   key, value    [num_tokens, num_kv_heads, head_dim]            same dtype
 *   slot_mapping  [num_tokens] int64, slot = block * B + row; negative = skip
 *   block_mapping [num_pairs, 2] int32, (src, dst) block ids
 * Query head h reads kv head h / (num_q_heads / num_kv_heads): contiguous groups (GQA).
 *
 * Supported shapes: head_dim in {64, 128}; block_size in {8, 16, 32};
 * num_q_heads a multiple of num_kv_heads.  Every pointer to q, out, caches, key and
 * value must be 16-byte aligned.
 *
 * Ownership: the caller owns every buffer.  The library allocates no device memory;
 * pa_decode's scratch is the caller's `workspace`.  Device calls are asynchronous on
 * `stream` (NULL = the legacy default stream) and return before the GPU work ends.
 *
 * Status codes: every int-returning call returns PA_OK (0) or a negative PA_ERR_*.
 * Argument errors are found on the host before anything is launched.  Errors that
 * only the device can see (a block id outside the pool, a context length < 1 or
 * > max_blocks_per_seq * B, a slot beyond the pool, a bad copy pair) make the kernel
 * skip that work item -- decode writes zeros for the affected sequence -- and set a
 * bit in a per-device error word that pa_get_device_error reads.  No kernel traps.
 */
#ifndef PA_H_
#define PA_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* PA_FP8_E4M3 names FP8 K/V blocks; it is accepted only where a call handles caches
 * alone (pa_copy_blocks, pa_swap_blocks).  The FP8 decode and cache write take the
 * 16-bit type of q / out / key / value instead. */
typedef enum { PA_FP16 = 0, PA_BF16 = 1, PA_FP8_E4M3 = 2 } pa_dtype;

enum {
  PA_OK = 0,
  PA_ERR_ARG = -1,            /* null pointer, unsupported shape or dtype, misalignment */
  PA_ERR_WORKSPACE = -2,      /* workspace missing or smaller than pa_decode_workspace_size */
  PA_ERR_CUDA = -3,           /* a CUDA runtime call failed (launch, attribute, copy) */
  PA_ERR_POOL_EXHAUSTED = -4, /* not enough free blocks; the pool is unchanged */
  PA_ERR_UNKNOWN_SEQ = -5,    /* sequence id not live (or already live, for a new id) */
  PA_ERR_WRONG_TIER = -6      /* sequence swapped out where a resident one is needed, or
                                 resident where a swapped-out one is needed */
};

/* Bits of the per-device error word (pa_get_device_error). */
#define PA_DEVERR_BAD_BLOCK   0x1u  /* decode: a used block-table entry is outside [0, num_blocks) */
#define PA_DEVERR_BAD_CONTEXT 0x2u  /* decode: context length < 1 or > max_blocks_per_seq * B */
#define PA_DEVERR_BAD_SLOT    0x4u  /* reshape_and_cache: slot >= num_blocks * B */
#define PA_DEVERR_BAD_PAIR    0x8u  /* copy_blocks / swap_blocks: a block id outside its pool */
#define PA_DEVERR_TIMEOUT     0x10u /* a bounded wait gave up (about 1 s; prefill pipeline, decode
                                         split-KV merge): output invalid */

/*
 * pa_reshape_and_cache -- write each new token's K and V rows into its cache slot.
 *
 * A new token's K/V row goes into the free slot of its sequence's last block; when
 * that block is full a fresh block from the free pool is appended to the table first
 * (chenyuan1125 "vllm-pagedattention", section 页表真正解开的…; horeb.top "vLLM
 * PagedAttention：大模型推理的显存管理革命", section 分配策略).  The host chooses the
 * slots (pa_pool_append_slot); this call only moves the bytes:
 *   k_cache[slot / B, h, slot % B, :] = key[i, h, :]   (and v_cache from value)
 * for every token i whose slot_mapping[i] >= 0.  Two tokens naming the same slot in
 * one call give an undefined winner.  Slots >= num_blocks * B are skipped and flagged
 * (PA_DEVERR_BAD_SLOT).  num_tokens == 0 is a no-op.
 */
int pa_reshape_and_cache(const void* key, const void* value, void* k_cache, void* v_cache,
                         const int64_t* slot_mapping, int num_tokens, int num_blocks,
                         int num_kv_heads, int head_dim, int block_size, pa_dtype dtype,
                         cudaStream_t stream);

/*
 * pa_decode -- single-query (decode) attention over paged K/V.
 *
 * For every sequence s and query head h (kv head g = h / G):
 *   z_t = scale * <q[s,h,:], K_s[t,g,:]>,  t < context_lens[s]
 *   out[s,h,:] = sum_t softmax(z)_t * V_s[t,g,:]
 * where K_s[t] = k_cache[block_tables[s][t / B], :, t % B, :] (same for V).  Scores,
 * the softmax and the weighted sum run block by block through the table
 * (daiw.org "Paged Attention", section 定义, Attention 内核; chenyuan1125, section
 * 页表真正解开的…).  Accumulation is fp32; the output is rounded to nearest-even.
 *
 * Work is split into equal shares of K/V stages (16 tokens; 32 over FP8 / INT4 blocks),
 * one share per SM, so a long sequence may be cut into pieces; the SM that finishes a
 * pair's last outstanding piece merges them with a log-sum-exp reduction (split-KV)
 * inside the same kernel, in a fixed order.  Cut points depend only on logical token
 * positions and the batch's context lengths, never on where blocks sit, so permuting
 * physical blocks (and the table with them) gives bit-identical output.
 *
 * workspace: device scratch of at least pa_decode_workspace_size(...) bytes for the
 * split pieces and their arrival counters, 16-byte aligned, owned by the caller.  Its
 * contents between calls do not matter: a counter left by another call (or never
 * written) is recognised by a tag that differs from call to call, and each merge leaves
 * its counter at zero, so calls replayed from a captured CUDA graph, which repeat their
 * tag, start from zero too.  Concurrent pa_decode calls must not share a workspace.
 * Returns PA_ERR_WORKSPACE if it is NULL or too small.  num_seqs == 0 is a no-op.
 *
 * Ordering: a launch is a programmatic dependent of the kernel before it in the stream.
 * It reads context_lens and block_tables (to plan its work) while that kernel drains,
 * and q, the caches and the workspace only after it has finished.  So block_tables and
 * context_lens must not be written by the kernel immediately before it in the stream
 * when that kernel lets its dependents start early (no kernel of this library writes
 * them; a plain copy or a kernel without programmatic launch is always safe).  The same
 * holds for every decode entry point below.
 */
int pa_decode(const void* q, const void* k_cache, const void* v_cache,
              const int32_t* block_tables, int max_blocks_per_seq,
              const int32_t* context_lens, int num_seqs, int num_q_heads, int num_kv_heads,
              int head_dim, int block_size, int num_blocks, float scale, void* out,
              void* workspace, size_t workspace_bytes, pa_dtype dtype, cudaStream_t stream);

/*
 * FP8 KV blocks.  Paging does not reduce the bytes the cache needs; quantising the cached
 * K/V does (daiw.org "Paged Attention", section 量化, callout; horeb.top, section 生态现状:
 * serving engines store KV in FP8 or INT4).  Format: each cache element is an E4M3 code
 * (1 sign, 4 exponent bits with bias 7, 3 mantissa bits; exponent field 0 = subnormals
 * m * 2^-9; no infinities; S.1111.111 is NaN; largest finite 448), in the same
 * [num_blocks][Hkv][B][d] layout, one byte per element.  One float32 scale per cache: a
 * code c means decode(c) * k_scale in the K cache and decode(c) * v_scale in the V cache.
 * Scales are the caller's (calibrated or fixed); both must be finite and > 0.
 */
/* Quantising cache write: k_cache[slot / B, h, slot % B, :] = E4M3(key[i, h, :] / k_scale)
 * (V likewise), the division in IEEE float32, rounding to nearest-even, magnitudes above
 * 448 clamped to 448.  key / value are fp16 or bf16 (`dtype`); other rules as
 * pa_reshape_and_cache. */
int pa_reshape_and_cache_fp8(const void* key, const void* value, void* k_cache, void* v_cache,
                             const int64_t* slot_mapping, int num_tokens, int num_blocks,
                             int num_kv_heads, int head_dim, int block_size, float k_scale,
                             float v_scale, pa_dtype dtype, cudaStream_t stream);
/* pa_decode over FP8 blocks: z_t = scale * k_scale * <q, decode(K codes)>, out = v_scale *
 * sum_t softmax(z)_t decode(V codes).  q and out are fp16 or bf16 (`dtype`).  The codes
 * are widened to f16 exactly and multiplied on the tensor cores in f16 (bf16 queries are
 * rounded to f16 for that product); accumulation fp32.  Same workspace, error and
 * determinism rules as pa_decode; there is no fused cache write for FP8 blocks. */
int pa_decode_fp8(const void* q, const void* k_cache, const void* v_cache,
                  const int32_t* block_tables, int max_blocks_per_seq,
                  const int32_t* context_lens, int num_seqs, int num_q_heads, int num_kv_heads,
                  int head_dim, int block_size, int num_blocks, float scale, float k_scale,
                  float v_scale, void* out, void* workspace, size_t workspace_bytes,
                  pa_dtype dtype, cudaStream_t stream);

/* One FP8 decode step in one call and one launch: each sequence's newest token (key_new /
 * value_new [num_seqs][Hkv][d], fp16 or bf16) is quantised with the arithmetic of
 * pa_reshape_and_cache_fp8 by the warp that computes the sequence's last stage, attended
 * from there and stored at position context_lens[s] - 1 through the table; caches and
 * output equal pa_reshape_and_cache_fp8 + pa_decode_fp8 bit for bit.  (A sequence whose
 * newest slot is invalid writes nothing; the decode flags it.) */
int pa_decode_append_fp8(const void* q, const void* key_new, const void* value_new,
                         void* k_cache, void* v_cache, const int32_t* block_tables,
                         int max_blocks_per_seq, const int32_t* context_lens, int num_seqs,
                         int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                         int num_blocks, float scale, float k_scale, float v_scale, void* out,
                         void* workspace, size_t workspace_bytes, pa_dtype dtype,
                         cudaStream_t stream);

/*
 * INT4 KV blocks (the other quantised format horeb.top, section 生态现状, names).  The
 * pages give no INT4 format; this one is symmetric integer quantisation with one scale
 * per cached row:
 *   codes   [num_blocks][Hkv][B][d/2] uint8: two 4-bit codes per byte, element 2i in the
 *           low nibble of byte i, each stored as u = c + 8 for a code c in [-7, 7];
 *   scales  [num_blocks][Hkv][B] float32, one per (block, kv head, row), K and V apart.
 * A row (one token of one kv head) means the values c_i * s.  All arrays 16-byte aligned,
 * owned by the caller.
 */
/* Quantising cache write: for each token i with slot = slot_mapping[i] >= 0 and each kv
 * head h, the row x = key[i, h, :] gets s = max_j |x_j| / 7 and c_j = x_j / s (both IEEE
 * float32 divisions) rounded to nearest-even and clamped to [-7, 7] (s = 0 and c = 0 for
 * an all-zero row); likewise value.  Inputs are finite fp16 or bf16 (`dtype`); other
 * rules as pa_reshape_and_cache. */
int pa_reshape_and_cache_int4(const void* key, const void* value, void* k_codes, void* v_codes,
                              float* k_scales, float* v_scales, const int64_t* slot_mapping,
                              int num_tokens, int num_blocks, int num_kv_heads, int head_dim,
                              int block_size, pa_dtype dtype, cudaStream_t stream);
/* pa_decode over INT4 blocks: z_t = scale * sK_t * <q, cK_t>, out = sum_t softmax(z)_t *
 * sV_t * cV_t.  q and out are fp16 or bf16 (`dtype`).  The codes are widened to f16
 * exactly and multiplied on the tensor cores in f16 (bf16 queries rounded to f16); each
 * token's K scale multiplies its fp32 scores, and each token's V scale multiplies its
 * softmax weight before that weight is rounded to f16 for P V (so V rows need
 * max|v| < 7 * 65504, and rows with max|v| below about 4e-4 lose precision to f16
 * subnormals).  Same workspace, error and determinism rules as pa_decode. */
int pa_decode_int4(const void* q, const void* k_codes, const void* v_codes, const float* k_scales,
                   const float* v_scales, const int32_t* block_tables, int max_blocks_per_seq,
                   const int32_t* context_lens, int num_seqs, int num_q_heads, int num_kv_heads,
                   int head_dim, int block_size, int num_blocks, float scale, void* out,
                   void* workspace, size_t workspace_bytes, pa_dtype dtype, cudaStream_t stream);
/* One INT4 decode step in one call and one launch: each sequence's newest token (key_new /
 * value_new [num_seqs][Hkv][d]) is quantised with the arithmetic of
 * pa_reshape_and_cache_int4 by the warp that computes its last stage, attended from there
 * and stored (codes and scales) at position context_lens[s] - 1 through the table; equal to
 * pa_reshape_and_cache_int4 + pa_decode_int4 bit for bit (a sequence whose newest slot is
 * invalid writes nothing and the decode flags it). */
int pa_decode_append_int4(const void* q, const void* key_new, const void* value_new,
                          void* k_codes, void* v_codes, float* k_scales, float* v_scales,
                          const int32_t* block_tables, int max_blocks_per_seq,
                          const int32_t* context_lens, int num_seqs, int num_q_heads,
                          int num_kv_heads, int head_dim, int block_size, int num_blocks,
                          float scale, void* out, void* workspace, size_t workspace_bytes,
                          pa_dtype dtype, cudaStream_t stream);
/* pa_copy_blocks for INT4 blocks: the codes and the scales of each pair (two launches). */
int pa_copy_blocks_int4(void* k_codes, void* v_codes, float* k_scales, float* v_scales,
                        const int32_t* block_mapping, int num_pairs, int num_blocks,
                        int num_kv_heads, int head_dim, int block_size, cudaStream_t stream);
/* pa_swap_blocks for INT4 blocks: codes and scales move together between two pools (one
 * of them may be pinned host memory); the same pair rules. */
int pa_swap_blocks_int4(const void* src_k, const void* src_v, const float* src_ks,
                        const float* src_vs, void* dst_k, void* dst_v, float* dst_ks,
                        float* dst_vs, const int32_t* block_mapping, int num_pairs,
                        int src_num_blocks, int dst_num_blocks, int num_kv_heads, int head_dim,
                        int block_size, cudaStream_t stream);

/*
 * pa_prefill -- causal multi-query attention of each sequence's newest tokens over its
 * paged context (a prompt from scratch, or a chunk of one).
 *
 * Sequence s owns query rows query_start[s] .. query_start[s+1]-1 of q: its newest
 * q_len_s = query_start[s+1] - query_start[s] tokens, at positions ctx_s - q_len_s ..
 * ctx_s - 1, whose K/V rows are already in the cache (write them first with
 * pa_reshape_and_cache).  The token at position p attends to positions 0 .. p:
 *   out[row, h, :] = sum_{t <= p} softmax(scale * <q[row, h, :], K_s[t, h / G, :]>) V_s[t, h / G, :]
 * with K_s[t] = k_cache[block_tables[s][t / B], :, t % B, :] (horeb.top "vLLM
 * PagedAttention：大模型推理的显存管理革命", section 分配策略: a prompt is allotted its
 * blocks at prefill; daiw.org "Paged Attention", section 回顾与衔接: the attention kernel
 * reads the block table).  Accumulation is fp32, the output rounded to nearest-even.
 *
 * q, out: [query_start[num_seqs], Hq, d] device, 16-byte aligned; query_start: int32
 * [num_seqs + 1] device, non-decreasing from 0; max_query_len: host bound on q_len_s
 * (the launch covers it; larger q_len_s are not computed).  Requires Hq / Hkv <= 64.
 * A sequence whose context is invalid (ctx < 1, ctx > T * B, or q_len_s > ctx_s) gets
 * zeros and PA_DEVERR_BAD_CONTEXT; a block id out of range gives zeros for the query
 * block that reads it and PA_DEVERR_BAD_BLOCK.  Uses no workspace.  A launch is a
 * programmatic dependent of the kernel before it in the stream.
 */
int pa_prefill(const void* q, const void* k_cache, const void* v_cache,
               const int32_t* block_tables, int max_blocks_per_seq,
               const int32_t* context_lens, const int32_t* query_start, int num_seqs,
               int max_query_len, int num_q_heads, int num_kv_heads, int head_dim,
               int block_size, int num_blocks, float scale, void* out, pa_dtype dtype,
               cudaStream_t stream);

/*
 * pa_decode_append -- one whole decode step in one kernel: the cache write of every
 * sequence's newest token followed by pa_decode over contexts that include it.
 *
 * key_new, value_new: [num_seqs, Hkv, d] device, row s = the token just produced by
 * sequence s, at its position ctx_s - 1, so its slot is
 * block_tables[s][(ctx_s - 1) / B] * B + (ctx_s - 1) % B (the slot formula of
 * pa_reshape_and_cache; chenyuan1125, section 页表真正解开的…: the new token goes into the
 * last block's free slot, then attention reads the context through the table).
 * Results -- out and both caches -- are bit-identical to pa_reshape_and_cache of those rows
 * into those slots followed by pa_decode with the same arguments.  The attention takes the
 * newest row from key_new/value_new, and the cache row is stored during the same kernel,
 * so that slot must not lie inside another sequence's context in the same call (true once
 * copy-on-write has given every written last block a single owner).  A sequence whose
 * context length or newest block id is invalid writes nothing and is flagged as in
 * pa_decode.  Other arguments, errors and the workspace are pa_decode's.
 */
int pa_decode_append(const void* q, const void* key_new, const void* value_new, void* k_cache,
                     void* v_cache, const int32_t* block_tables, int max_blocks_per_seq,
                     const int32_t* context_lens, int num_seqs, int num_q_heads,
                     int num_kv_heads, int head_dim, int block_size, int num_blocks, float scale,
                     void* out, void* workspace, size_t workspace_bytes, pa_dtype dtype,
                     cudaStream_t stream);

/*
 * pa_decode_fixed_scratch -- pa_decode for callers that cannot allocate device memory.
 *
 * The pages have no counterpart to this call; it exists for library users.  Some callers
 * may not call cudaMalloc at all -- a server that gave nearly all HBM to the KV block pool
 * up front, or a host framework that owns every device buffer -- and so cannot supply
 * pa_decode's workspace.  This call takes the same arguments minus the workspace and uses
 * a fixed 32 MiB scratch array built into the library instead (held on every GPU that
 * loads the library until the process exits).  It allocates nothing.
 *   - Every call on a device shares that scratch and leaves its contents behind; nothing in
 *     it needs to start at zero.  Calls whose GPU work overlaps (unordered streams) race on
 *     it and give undefined output.
 *   - The first call on a device looks up the scratch's device address there; make that
 *     first call before any stream capture begins.
 *   - A device and head shape needing more than 32 MiB of decode scratch (more than about
 *     250 SMs at 16 query heads per kv head and head_dim 128) gets PA_ERR_WORKSPACE and
 *     nothing is launched.
 *   - q must be device memory of the current device (the scratch is per device); a q
 *     elsewhere gets PA_ERR_ARG.  Other errors are pa_decode's.
 */
int pa_decode_fixed_scratch(const void* q, const void* k_cache, const void* v_cache,
                            const int32_t* block_tables, int max_blocks_per_seq,
                            const int32_t* context_lens, int num_seqs, int num_q_heads,
                            int num_kv_heads, int head_dim, int block_size, int num_blocks,
                            float scale, void* out, pa_dtype dtype, cudaStream_t stream);

/*
 * pa_decode_timeline -- diagnostics: time the phases of 16-bit decode launches.
 *
 * The pages have no counterpart; it exists to measure where a launch's time goes.  While
 * a buffer is set, every decode launch made by this host thread (pa_decode,
 * pa_decode_append, pa_decode_fixed_scratch) runs a copy of the kernel in which lane 0 of
 * each warp writes three %globaltimer readings (ns) into the buffer.  That works for
 * 16-bit blocks at head_dim 128 with at most 8 query heads per kv head.  Launches made
 * without a buffer run the kernel without that code.  The layout is [cta][warp][k]
 * unsigned long long with 8 warps a CTA, and k is:
 *   0  the programmatic wait on the previous kernel released,
 *   1  the warp's streaming done (before the cut pieces are counted in),
 *   2  its end (after any merge).
 * A CTA with no work writes nothing, so zero the buffer first.  buffer is device memory of
 * at least SM count x 8 x 3 x 8 bytes (29 184 bytes on 152 SMs).  While a buffer is set,
 * a decode launch returns PA_ERR_ARG and launches nothing if the buffer is smaller than
 * that, if the blocks are FP8 or INT4, or if the shape is another one.  NULL clears the
 * setting.  The caller owns the buffer, and outputs are unaffected.  Returns PA_ERR_ARG
 * for a non-null buffer that is not 8-byte aligned.
 */
int pa_decode_timeline(void* buffer, size_t bytes);

/* Bytes of workspace pa_decode needs on the current device for these head counts.
 * It depends on the device's SM count and the head shape only, not on the batch
 * (152 SMs: 5.1 MB for 32 query / 8 kv heads at head_dim 128, at most about 20 MB). */
size_t pa_decode_workspace_size(int num_q_heads, int num_kv_heads, int head_dim);

/*
 * pa_copy_blocks -- copy whole physical blocks (every kv head, every row) of both
 * caches: k_cache[dst] = k_cache[src], v_cache[dst] = v_cache[src] for each pair.
 *
 * This is the copy behind copy-on-write: a branch that must write into a last block
 * still shared with other sequences first copies it, then remaps and writes; full old
 * blocks stay shared (chenyuan1125, section 一块内存，如何安全地属于多条序列; horeb.top,
 * section 内存共享：写时复制).  block_mapping is device memory.  Pairs must not alias
 * (distinct dst, no dst also a src); pa_check_block_mapping checks a host copy.  A pair
 * with an id outside [0, num_blocks) is skipped and flagged (PA_DEVERR_BAD_PAIR).
 */
int pa_copy_blocks(void* k_cache, void* v_cache, const int32_t* block_mapping, int num_pairs,
                   int num_blocks, int num_kv_heads, int head_dim, int block_size,
                   pa_dtype dtype, cudaStream_t stream);

/*
 * pa_swap_blocks -- copy whole blocks from one pool to another:
 *   dst_k[d] = src_k[s], dst_v[d] = src_v[s]  for each pair (s, d) of block_mapping.
 *
 * This moves a preempted request's blocks to CPU memory (swap-out) and back (swap-in);
 * the block table is what makes the move a plain block copy (aiqz.cc "vLLM
 * PagedAttention engine", section 连续批处理：随到随走的新秩序).  pa_pool_swap_out /
 * pa_pool_swap_in plan the pairs.
 *
 * Pools: src [src_num_blocks, Hkv, B, d], dst [dst_num_blocks, Hkv, B, d], same dtype.
 * Each of the five pointers may be device memory or page-locked host memory registered
 * with CUDA (cudaHostAlloc, cudaMallocHost, cudaHostRegister; a pinned torch tensor):
 * the GPU reads and writes host memory directly (over NVLink-C2C on GB300), so one
 * kernel launch moves every pair.  Anything else (pageable host memory) is PA_ERR_ARG.
 * block_mapping is int32 [num_pairs, 2].  Destination ids must be distinct and the two
 * pools must not overlap.  A pair with an id outside its pool is skipped and flagged
 * (PA_DEVERR_BAD_PAIR).  num_pairs == 0 is a no-op.
 */
int pa_swap_blocks(const void* src_k, const void* src_v, void* dst_k, void* dst_v,
                   const int32_t* block_mapping, int num_pairs, int src_num_blocks,
                   int dst_num_blocks, int num_kv_heads, int head_dim, int block_size,
                   pa_dtype dtype, cudaStream_t stream);

/* Host-side check of a copy_blocks pair list (host memory): PA_OK, or PA_ERR_ARG when an
 * id is outside [0, num_blocks), a dst repeats, or a dst is also a src. */
int pa_check_block_mapping(const int32_t* host_block_mapping, int num_pairs, int num_blocks);

/* Synchronise `stream`, then read and clear the current device's error word. */
int pa_get_device_error(cudaStream_t stream, uint32_t* flags_out);

/* Human-readable name of a status code (static string). */
const char* pa_status_string(int status);

/*
 * Host block pool: free list, reference counts, fork and copy-on-write planning.
 *
 * Blocks leave the head of an ordered free list and return to its tail (aiqz.cc,
 * section Python 演示).  Prefill takes ceil(n / B) blocks; decode takes a new block
 * every B tokens; a finished sequence returns its blocks (horeb.top, section 分配策略).
 * A block shared by several sequences is reclaimed only when its reference count
 * reaches zero (daiw.org "Paged Attention", section 量化).  When a sequence must write
 * into a partly filled last block whose count is above one, the pool plans a copy: it
 * takes a new block, moves this sequence's table entry to it and returns the (src, dst)
 * pair, which the caller copies with pa_copy_blocks before writing (chenyuan1125,
 * section 一块内存…).  An operation that cannot get every block it needs changes
 * nothing and returns PA_ERR_POOL_EXHAUSTED (daiw.org, section 速查卡: an exhausted pool
 * rejects new requests instead of failing).  Host memory only; not thread-safe.
 *
 * A second pool of CPU blocks (pa_pool_create_tiered) backs preemption: a group of
 * resident sequences is swapped out whole and later swapped back in (aiqz.cc, section
 * 连续批处理：随到随走的新秩序).  Each distinct block of the group's tables (sequences in
 * the order given, tables in order, first appearance) takes one block from the head of
 * the other pool's free list and carries the group's references to it; the old block
 * loses them and, at zero, returns to its pool's tail in that order.  The tables are
 * rewritten to the new ids.  A swapped-out sequence can be freed or swapped in; grow,
 * fork and pa_pool_slots return PA_ERR_WRONG_TIER.
 */
typedef struct pa_pool pa_pool;

/* initial_free_order: NULL for 0..num_blocks-1, else a permutation of it (host).
 * Returns NULL on a bad argument or allocation failure. */
pa_pool* pa_pool_create(int num_blocks, int block_size, const int32_t* initial_free_order);
/* The same with a CPU pool of num_cpu_blocks (>= 0) blocks, free order cpu_free_order
 * (NULL for 0..num_cpu_blocks-1, else a permutation of it). */
pa_pool* pa_pool_create_tiered(int num_blocks, int block_size, const int32_t* initial_free_order,
                               int num_cpu_blocks, const int32_t* cpu_free_order);
void pa_pool_destroy(pa_pool* pool);
/* Prefill: a new sequence holding n_tokens tokens in ceil(n_tokens / B) blocks. */
int pa_pool_allocate(pa_pool* pool, int64_t seq_id, int n_tokens);
/* Reserve the next token's slot.  Returns 0, or 1 when a copy is planned (then
 * *cow_src, *cow_dst name the blocks to copy before writing), or a negative error. */
int pa_pool_append_slot(pa_pool* pool, int64_t seq_id, int64_t* slot_out, int32_t* cow_src,
                        int32_t* cow_dst);
/* The child shares every block of the parent (reference counts + 1). */
int pa_pool_fork(pa_pool* pool, int64_t parent_id, int64_t child_id);
/* End a sequence; blocks whose count reaches zero go to the free-list tail in table order. */
int pa_pool_free(pa_pool* pool, int64_t seq_id);
/* Copy up to `cap` table entries into out; returns the table length or an error. */
int pa_pool_block_table(const pa_pool* pool, int64_t seq_id, int32_t* out, int cap);
/* Tokens held by the sequence, or an error. */
int pa_pool_context_len(const pa_pool* pool, int64_t seq_id);
/* Slots of logical tokens [first, first + count) of the sequence (all < context_len). */
int pa_pool_slots(const pa_pool* pool, int64_t seq_id, int first, int count, int64_t* slots_out);
int pa_pool_num_free(const pa_pool* pool);
/* Copy up to `cap` free-list entries, head first; returns the free-list length. */
int pa_pool_free_list(const pa_pool* pool, int32_t* out, int cap);
/* Reference count of a block, or PA_ERR_ARG for an id outside the pool. */
int pa_pool_refcount(const pa_pool* pool, int32_t block);
/* Swap a group of n distinct resident sequences out to the CPU pool.  Writes the
 * (device block, CPU block) pairs to pairs_out [cap][2] and returns their number, or an
 * error (PA_ERR_ARG for a repeated id or cap too small, PA_ERR_UNKNOWN_SEQ,
 * PA_ERR_WRONG_TIER, PA_ERR_POOL_EXHAUSTED); on error nothing changes.  The caller then
 * copies the pairs with pa_swap_blocks (device pool -> CPU pool). */
int pa_pool_swap_out(pa_pool* pool, const int64_t* seq_ids, int n, int32_t* pairs_out, int cap);
/* The mirror image: (CPU block, device block) pairs, copied CPU pool -> device pool. */
int pa_pool_swap_in(pa_pool* pool, const int64_t* seq_ids, int n, int32_t* pairs_out, int cap);
/* 1 if the sequence is swapped out, 0 if resident, or PA_ERR_UNKNOWN_SEQ. */
int pa_pool_is_swapped(const pa_pool* pool, int64_t seq_id);
int pa_pool_num_free_cpu(const pa_pool* pool);
int pa_pool_cpu_free_list(const pa_pool* pool, int32_t* out, int cap);
int pa_pool_cpu_refcount(const pa_pool* pool, int32_t block);

/*
 * Automatic prefix caching.  A full block is named by its parent's digest, its tokens and
 * the request's extra keys, so a prompt that starts with blocks already in the pool
 * reuses their K/V and skips that part of prefill (chenyuan1125, section
 * 一块内存，如何安全地属于多条序列); `extra` (a tenant's cache salt, an adapter id, ...)
 * keeps requests that must not share apart (same page, section 分页不是免费午餐).
 * Digest of full block i (SHA-256, FIPS 180-4; integers little-endian):
 *   SHA-256(digest_{i-1} || B as u32 || tokens[iB .. iB+B-1] as i32 || extra_len as u32
 *           || extra),   digest_{-1} = 32 zero bytes.
 * The lookup walks the prompt's full blocks in order and stops at the first miss.  A hit
 * adds a reference to the cached block (taking it out of the free list if its count was
 * zero); the rest of the prompt gets blocks from the head of the free list, and each full
 * block among them is registered under its digest unless the digest already names a
 * block.  A cached block at count zero stays cached in the free list, so the free-list
 * order is the eviction order; any block taken from the head loses its digest.  Partly
 * filled blocks and blocks filled by decode are not registered.
 */
/* Prefill with prefix caching: a new sequence holding tokens[0 .. n_tokens-1] (host
 * int32).  *cached_tokens_out (may be NULL) receives the number of leading tokens whose
 * K/V the reused blocks already hold (a multiple of B); the caller computes and writes
 * the rest.  Errors as pa_pool_allocate; on error nothing changes. */
int pa_pool_allocate_prefix(pa_pool* pool, int64_t seq_id, const int32_t* tokens, int n_tokens,
                            const uint8_t* extra, int extra_len, int* cached_tokens_out);
/* A scheduler step's prompts in one call: requests r = 0..n-1 with ids seq_ids[r], tokens
 * tokens[token_start[r] .. token_start[r+1]-1] and extra bytes extras[extra_start[r] ..
 * extra_start[r+1]-1] (extras NULL: none), placed in order exactly as n calls of
 * pa_pool_allocate_prefix would.  The digest chains of different requests are computed in
 * parallel on a small pool of host threads (the library's own; batch calls are serialised
 * on it).  Outputs: cached_out[n]; slots_out (may be NULL) the slots of every request's
 * uncached tokens, request after request (what pa_reshape_and_cache takes for the new
 * rows); tables_out (may be NULL) [n][table_width] block tables padded with 0.
 * token_start and extra_start must start at 0 or above and never decrease.  A negative
 * start, a decreasing offset, a span longer than INT_MAX or a table wider than
 * table_width is PA_ERR_ARG before anything changes.  On a later error the requests
 * before the failing one stay allocated: *n_done (may be NULL) says how many. */
/* The table width a batch of n requests needs (tokens token_start[r] .. token_start[r+1]-1
 * each): the largest number of blocks one of them takes, ceil(tokens / B); PA_ERR_ARG for
 * a negative start or a decreasing offset. */
int pa_pool_table_width(const pa_pool* pool, int n, const int64_t* token_start);
int pa_pool_allocate_prefix_batch(pa_pool* pool, int n, const int64_t* seq_ids,
                                  const int32_t* tokens, const int64_t* token_start,
                                  const uint8_t* extras, const int64_t* extra_start,
                                  int* cached_out, int64_t* slots_out, int32_t* tables_out,
                                  int table_width, int* n_done);
/* The same placement from digests computed earlier (pa_prefix_block_hashes when a request
 * arrives, say, so that hashing stays off the scheduling step): request r holds
 * n_tokens[r] tokens, and `digests` holds the 32-byte digests of every request's
 * n_tokens[r] / B full blocks, request after request.  Results equal
 * pa_pool_allocate_prefix_batch on the tokens those digests came from. */
int pa_pool_allocate_hashed_batch(pa_pool* pool, int n, const int64_t* seq_ids,
                                  const int32_t* n_tokens, const uint8_t* digests,
                                  int* cached_out, int64_t* slots_out, int32_t* tables_out,
                                  int table_width, int* n_done);
/* pa_pool_free of n sequences in order; stops at the first error. */
int pa_pool_free_batch(pa_pool* pool, const int64_t* seq_ids, int n);
/* Number of blocks registered under a digest (in use or waiting in the free list). */
int pa_pool_num_cached(const pa_pool* pool);
/* 1 and the block's 32-byte digest, 0 if the block has none, or PA_ERR_ARG. */
int pa_pool_block_digest(const pa_pool* pool, int32_t block, uint8_t* digest_out);
/* The digests of the n_tokens / B full blocks of a token list into digests_out
 * [cap][32]; returns their number (pure host function). */
int pa_prefix_block_hashes(const int32_t* tokens, int n_tokens, int block_size,
                           const uint8_t* extra, int extra_len, uint8_t* digests_out, int cap);
/* SHA-256 of `len` bytes (FIPS 180-4) into digest_out[32]. */
int pa_sha256(const void* data, size_t len, uint8_t* digest_out);

#ifdef __cplusplus
}
#endif
#endif /* PA_H_ */
