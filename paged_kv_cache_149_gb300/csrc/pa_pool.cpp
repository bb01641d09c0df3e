// Host block pool: ordered free list, per-block reference counts, fork and
// copy-on-write planning.  Blocks leave the head of the free list and return to its
// tail (aiqz.cc "vLLM PagedAttention engine", section Python 演示); prefill takes
// ceil(n / B) blocks and decode one block every B tokens (horeb.top, section
// 分配策略); a shared block is reclaimed at reference count zero (daiw.org "Paged
// Attention", section 量化); a write into a shared, partly filled last block copies it
// first (chenyuan1125 "vllm-pagedattention", section 一块内存，如何安全地属于多条序列).
// Preemption moves a request's blocks whole into CPU memory and back (aiqz.cc, section
// 连续批处理：随到随走的新秩序): a second pool of CPU blocks follows the same rules, and
// swap_out / swap_in plan the block moves that pa_swap_blocks then performs.
//
// Each pool's free list is a ring buffer of capacity num_blocks: every block id is either
// in the ring or referenced by at least one table of that pool, so the ring never
// overflows.
#include <cstdint>
#include <cstring>
#include <new>
#include <unordered_map>
#include <vector>

#include "../../include/pa.h"

namespace {

struct SeqState {
  std::vector<int32_t> table;  // block ids of the pool the sequence lives in
  int64_t ctx = 0;
  bool swapped = false;        // true: the ids are CPU-pool ids
};

// One pool of blocks: ordered free list (ring) and reference counts.
struct Tier {
  int num_blocks = 0;
  std::vector<int32_t> ring;  // free list; head at `head`, `nfree` entries
  int head = 0;
  int nfree = 0;
  std::vector<int32_t> refcount;

  bool init(int n, const int32_t* order) {
    num_blocks = n;
    ring.resize(n);
    refcount.assign(n, 0);
    std::vector<char> seen(n, 0);
    for (int i = 0; i < n; ++i) {
      const int32_t b = order ? order[i] : i;
      if (b < 0 || b >= n || seen[b]) return false;
      seen[b] = 1;
      ring[i] = b;
    }
    nfree = n;
    return true;
  }
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

}  // namespace

struct pa_pool {
  int block_size = 0;
  Tier gpu, cpu;
  std::unordered_map<int64_t, SeqState> seqs;
};

extern "C" {

pa_pool* pa_pool_create_tiered(int num_blocks, int block_size, const int32_t* initial_free_order,
                               int num_cpu_blocks, const int32_t* cpu_free_order) {
  if (num_blocks <= 0 || block_size <= 0 || num_cpu_blocks < 0) return nullptr;
  pa_pool* p = new (std::nothrow) pa_pool();
  if (!p) return nullptr;
  try {
    p->block_size = block_size;
    if (!p->gpu.init(num_blocks, initial_free_order) ||
        !p->cpu.init(num_cpu_blocks, cpu_free_order)) {
      delete p;
      return nullptr;
    }
  } catch (...) {
    delete p;
    return nullptr;
  }
  return p;
}

pa_pool* pa_pool_create(int num_blocks, int block_size, const int32_t* initial_free_order) {
  return pa_pool_create_tiered(num_blocks, block_size, initial_free_order, 0, nullptr);
}

void pa_pool_destroy(pa_pool* pool) { delete pool; }

int pa_pool_allocate(pa_pool* pool, int64_t seq_id, int n_tokens) {
  if (!pool || n_tokens < 0) return PA_ERR_ARG;
  if (pool->seqs.count(seq_id)) return PA_ERR_UNKNOWN_SEQ;
  int64_t need = (static_cast<int64_t>(n_tokens) + pool->block_size - 1) / pool->block_size;
  if (need > pool->gpu.nfree) return PA_ERR_POOL_EXHAUSTED;
  SeqState st;
  st.table.reserve(static_cast<size_t>(need) + 1);
  for (int64_t i = 0; i < need; ++i) st.table.push_back(pool->gpu.pop());
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
  if (st.swapped) return PA_ERR_WRONG_TIER;
  const int64_t t = st.ctx;
  const int bs = pool->block_size;
  Tier& g = pool->gpu;
  int planned = 0;
  if (t % bs == 0) {
    // The last block is full (or there is none): open a fresh block.
    if (g.nfree < 1) return PA_ERR_POOL_EXHAUSTED;
    st.table.push_back(g.pop());
  } else if (g.refcount[st.table.back()] > 1) {
    // The partly filled last block is shared: copy it before writing.
    if (g.nfree < 1) return PA_ERR_POOL_EXHAUSTED;
    if (!cow_src || !cow_dst) return PA_ERR_ARG;
    int32_t old_b = st.table.back();
    int32_t new_b = g.pop();
    g.refcount[old_b] -= 1;
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
  if (it->second.swapped) return PA_ERR_WRONG_TIER;
  SeqState child = it->second;  // copy of the table and the token count
  for (int32_t b : child.table) pool->gpu.refcount[b] += 1;
  pool->seqs.emplace(child_id, std::move(child));
  return PA_OK;
}

int pa_pool_free(pa_pool* pool, int64_t seq_id) {
  if (!pool) return PA_ERR_ARG;
  auto it = pool->seqs.find(seq_id);
  if (it == pool->seqs.end()) return PA_ERR_UNKNOWN_SEQ;
  Tier& t = it->second.swapped ? pool->cpu : pool->gpu;
  for (int32_t b : it->second.table) {
    if (--t.refcount[b] == 0) t.push(b);
  }
  pool->seqs.erase(it);
  return PA_OK;
}

// Move a group of sequences to the other pool.  All checks come before any change.
static int pool_move(pa_pool* pool, const int64_t* seq_ids, int n, int32_t* pairs_out, int cap,
                     bool to_cpu) {
  if (!pool || n < 0 || (n > 0 && !seq_ids) || cap < 0) return PA_ERR_ARG;
  {
    std::unordered_map<int64_t, char> seen;
    for (int i = 0; i < n; ++i)
      if (!seen.emplace(seq_ids[i], 1).second) return PA_ERR_ARG;
  }
  std::vector<SeqState*> group;
  group.reserve(static_cast<size_t>(n));
  for (int i = 0; i < n; ++i) {
    auto it = pool->seqs.find(seq_ids[i]);
    if (it == pool->seqs.end()) return PA_ERR_UNKNOWN_SEQ;
    if (it->second.swapped == to_cpu) return PA_ERR_WRONG_TIER;
    group.push_back(&it->second);
  }
  Tier& src = to_cpu ? pool->gpu : pool->cpu;
  Tier& dst = to_cpu ? pool->cpu : pool->gpu;
  // distinct blocks in order of first appearance, with the group's references to each
  std::unordered_map<int32_t, int> index;
  std::vector<int32_t> blocks;
  std::vector<int32_t> refs;
  for (SeqState* st : group)
    for (int32_t b : st->table) {
      auto ins = index.emplace(b, static_cast<int>(blocks.size()));
      if (ins.second) {
        blocks.push_back(b);
        refs.push_back(1);
      } else {
        refs[ins.first->second] += 1;
      }
    }
  const int m = static_cast<int>(blocks.size());
  if (m > dst.nfree) return PA_ERR_POOL_EXHAUSTED;
  if (m > cap || (m > 0 && !pairs_out)) return PA_ERR_ARG;
  std::vector<int32_t> moved(static_cast<size_t>(m));
  for (int i = 0; i < m; ++i) {
    moved[i] = dst.pop();
    dst.refcount[moved[i]] = refs[i];
    src.refcount[blocks[i]] -= refs[i];
    if (src.refcount[blocks[i]] == 0) src.push(blocks[i]);
    pairs_out[2 * i] = blocks[i];
    pairs_out[2 * i + 1] = moved[i];
  }
  for (SeqState* st : group) {
    for (int32_t& b : st->table) b = moved[index[b]];
    st->swapped = to_cpu;
  }
  return m;
}

int pa_pool_swap_out(pa_pool* pool, const int64_t* seq_ids, int n, int32_t* pairs_out, int cap) {
  return pool_move(pool, seq_ids, n, pairs_out, cap, true);
}

int pa_pool_swap_in(pa_pool* pool, const int64_t* seq_ids, int n, int32_t* pairs_out, int cap) {
  return pool_move(pool, seq_ids, n, pairs_out, cap, false);
}

int pa_pool_is_swapped(const pa_pool* pool, int64_t seq_id) {
  if (!pool) return PA_ERR_ARG;
  auto it = pool->seqs.find(seq_id);
  if (it == pool->seqs.end()) return PA_ERR_UNKNOWN_SEQ;
  return it->second.swapped ? 1 : 0;
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
  if (st.swapped) return PA_ERR_WRONG_TIER;
  if (static_cast<int64_t>(first) + count > st.ctx) return PA_ERR_ARG;
  const int bs = pool->block_size;
  for (int i = 0; i < count; ++i) {
    int64_t t = static_cast<int64_t>(first) + i;
    slots_out[i] = static_cast<int64_t>(st.table[t / bs]) * bs + t % bs;
  }
  return PA_OK;
}

static int tier_free_list(const Tier& t, int32_t* out, int cap) {
  if (cap > 0 && !out) return PA_ERR_ARG;
  int m = t.nfree < cap ? t.nfree : cap;
  for (int i = 0; i < m; ++i) out[i] = t.ring[(t.head + i) % t.num_blocks];
  return t.nfree;
}

int pa_pool_num_free(const pa_pool* pool) { return pool ? pool->gpu.nfree : PA_ERR_ARG; }

int pa_pool_free_list(const pa_pool* pool, int32_t* out, int cap) {
  return pool ? tier_free_list(pool->gpu, out, cap) : PA_ERR_ARG;
}

int pa_pool_refcount(const pa_pool* pool, int32_t block) {
  if (!pool || block < 0 || block >= pool->gpu.num_blocks) return PA_ERR_ARG;
  return pool->gpu.refcount[block];
}

int pa_pool_num_free_cpu(const pa_pool* pool) { return pool ? pool->cpu.nfree : PA_ERR_ARG; }

int pa_pool_cpu_free_list(const pa_pool* pool, int32_t* out, int cap) {
  return pool ? tier_free_list(pool->cpu, out, cap) : PA_ERR_ARG;
}

int pa_pool_cpu_refcount(const pa_pool* pool, int32_t block) {
  if (!pool || block < 0 || block >= pool->cpu.num_blocks) return PA_ERR_ARG;
  return pool->cpu.refcount[block];
}

}  // extern "C"
