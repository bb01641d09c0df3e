// Host block pool: ordered free list, per-block reference counts, fork and
// copy-on-write planning.  Blocks leave the head of the free list and return to its
// tail (aiqz.cc "vLLM PagedAttention engine", section Python 演示); prefill takes
// ceil(n / B) blocks and decode one block every B tokens (horeb.top, section
// 分配策略); a shared block is reclaimed at reference count zero (daiw.org "Paged
// Attention", section 量化); a write into a shared, partly filled last block copies it
// first (chenyuan1125 "vllm-pagedattention", section 一块内存，如何安全地属于多条序列).
//
// The free list is a ring buffer of capacity num_blocks: every block id is either in
// the ring or referenced by at least one table, so the ring never overflows.
#include <cstdint>
#include <cstring>
#include <new>
#include <unordered_map>
#include <vector>

#include "../../include/pa.h"

namespace {

struct SeqState {
  std::vector<int32_t> table;
  int64_t ctx = 0;
};

}  // namespace

struct pa_pool {
  int num_blocks = 0;
  int block_size = 0;
  std::vector<int32_t> ring;  // free list; head at `head`, `nfree` entries
  int head = 0;
  int nfree = 0;
  std::vector<int32_t> refcount;
  std::unordered_map<int64_t, SeqState> seqs;

  int32_t pop() {
    int32_t b = ring[head];
    head = (head + 1) % num_blocks;
    --nfree;
    refcount[b] = 1;
    return b;
  }
  void push(int32_t b) {
    ring[(head + nfree) % num_blocks] = b;
    ++nfree;
  }
};

extern "C" {

pa_pool* pa_pool_create(int num_blocks, int block_size, const int32_t* initial_free_order) {
  if (num_blocks <= 0 || block_size <= 0) return nullptr;
  pa_pool* p = new (std::nothrow) pa_pool();
  if (!p) return nullptr;
  try {
    p->num_blocks = num_blocks;
    p->block_size = block_size;
    p->ring.resize(num_blocks);
    p->refcount.assign(num_blocks, 0);
    std::vector<char> seen(num_blocks, 0);
    for (int i = 0; i < num_blocks; ++i) {
      int32_t b = initial_free_order ? initial_free_order[i] : i;
      if (b < 0 || b >= num_blocks || seen[b]) {
        delete p;
        return nullptr;
      }
      seen[b] = 1;
      p->ring[i] = b;
    }
    p->nfree = num_blocks;
  } catch (...) {
    delete p;
    return nullptr;
  }
  return p;
}

void pa_pool_destroy(pa_pool* pool) { delete pool; }

int pa_pool_allocate(pa_pool* pool, int64_t seq_id, int n_tokens) {
  if (!pool || n_tokens < 0) return PA_ERR_ARG;
  if (pool->seqs.count(seq_id)) return PA_ERR_UNKNOWN_SEQ;
  int64_t need = (static_cast<int64_t>(n_tokens) + pool->block_size - 1) / pool->block_size;
  if (need > pool->nfree) return PA_ERR_POOL_EXHAUSTED;
  SeqState st;
  st.table.reserve(static_cast<size_t>(need) + 1);
  for (int64_t i = 0; i < need; ++i) st.table.push_back(pool->pop());
  st.ctx = n_tokens;
  pool->seqs.emplace(seq_id, std::move(st));
  return PA_OK;
}

int pa_pool_append_slot(pa_pool* pool, int64_t seq_id, int64_t* slot_out, int32_t* cow_src,
                        int32_t* cow_dst) {
  if (!pool || !slot_out) return PA_ERR_ARG;
  auto it = pool->seqs.find(seq_id);
  if (it == pool->seqs.end()) return PA_ERR_UNKNOWN_SEQ;
  SeqState& st = it->second;
  const int64_t t = st.ctx;
  const int bs = pool->block_size;
  int planned = 0;
  if (t % bs == 0) {
    // The last block is full (or there is none): open a fresh block.
    if (pool->nfree < 1) return PA_ERR_POOL_EXHAUSTED;
    st.table.push_back(pool->pop());
  } else if (pool->refcount[st.table.back()] > 1) {
    // The partly filled last block is shared: copy it before writing.
    if (pool->nfree < 1) return PA_ERR_POOL_EXHAUSTED;
    if (!cow_src || !cow_dst) return PA_ERR_ARG;
    int32_t old_b = st.table.back();
    int32_t new_b = pool->pop();
    pool->refcount[old_b] -= 1;
    st.table.back() = new_b;
    *cow_src = old_b;
    *cow_dst = new_b;
    planned = 1;
  }
  st.ctx = t + 1;
  *slot_out = static_cast<int64_t>(st.table[t / bs]) * bs + t % bs;
  return planned;
}

int pa_pool_fork(pa_pool* pool, int64_t parent_id, int64_t child_id) {
  if (!pool) return PA_ERR_ARG;
  auto it = pool->seqs.find(parent_id);
  if (it == pool->seqs.end() || pool->seqs.count(child_id)) return PA_ERR_UNKNOWN_SEQ;
  SeqState child = it->second;  // copy of the table and the token count
  for (int32_t b : child.table) pool->refcount[b] += 1;
  pool->seqs.emplace(child_id, std::move(child));
  return PA_OK;
}

int pa_pool_free(pa_pool* pool, int64_t seq_id) {
  if (!pool) return PA_ERR_ARG;
  auto it = pool->seqs.find(seq_id);
  if (it == pool->seqs.end()) return PA_ERR_UNKNOWN_SEQ;
  for (int32_t b : it->second.table) {
    if (--pool->refcount[b] == 0) pool->push(b);
  }
  pool->seqs.erase(it);
  return PA_OK;
}

int pa_pool_block_table(const pa_pool* pool, int64_t seq_id, int32_t* out, int cap) {
  if (!pool || (cap > 0 && !out)) return PA_ERR_ARG;
  auto it = pool->seqs.find(seq_id);
  if (it == pool->seqs.end()) return PA_ERR_UNKNOWN_SEQ;
  const std::vector<int32_t>& t = it->second.table;
  int n = static_cast<int>(t.size());
  int m = n < cap ? n : cap;
  if (m > 0) std::memcpy(out, t.data(), sizeof(int32_t) * m);
  return n;
}

int pa_pool_context_len(const pa_pool* pool, int64_t seq_id) {
  if (!pool) return PA_ERR_ARG;
  auto it = pool->seqs.find(seq_id);
  if (it == pool->seqs.end()) return PA_ERR_UNKNOWN_SEQ;
  return static_cast<int>(it->second.ctx);
}

int pa_pool_slots(const pa_pool* pool, int64_t seq_id, int first, int count, int64_t* slots_out) {
  if (!pool || first < 0 || count < 0 || (count > 0 && !slots_out)) return PA_ERR_ARG;
  auto it = pool->seqs.find(seq_id);
  if (it == pool->seqs.end()) return PA_ERR_UNKNOWN_SEQ;
  const SeqState& st = it->second;
  if (static_cast<int64_t>(first) + count > st.ctx) return PA_ERR_ARG;
  const int bs = pool->block_size;
  for (int i = 0; i < count; ++i) {
    int64_t t = static_cast<int64_t>(first) + i;
    slots_out[i] = static_cast<int64_t>(st.table[t / bs]) * bs + t % bs;
  }
  return PA_OK;
}

int pa_pool_num_free(const pa_pool* pool) { return pool ? pool->nfree : PA_ERR_ARG; }

int pa_pool_free_list(const pa_pool* pool, int32_t* out, int cap) {
  if (!pool || (cap > 0 && !out)) return PA_ERR_ARG;
  int m = pool->nfree < cap ? pool->nfree : cap;
  for (int i = 0; i < m; ++i) out[i] = pool->ring[(pool->head + i) % pool->num_blocks];
  return pool->nfree;
}

int pa_pool_refcount(const pa_pool* pool, int32_t block) {
  if (!pool || block < 0 || block >= pool->num_blocks) return PA_ERR_ARG;
  return pool->refcount[block];
}

}  // extern "C"
