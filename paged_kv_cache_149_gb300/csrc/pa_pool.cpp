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
// Automatic prefix caching makes full blocks findable by content: a block is named by
// its parent block's digest, its tokens and the request's extra keys (adapter, inputs,
// cache salt), and a new prompt that starts with the same blocks reuses their K/V
// (chenyuan1125, section 一块内存，如何安全地属于多条序列); a salt keeps tenants apart
// (same page, section 分页不是免费午餐).  Digests are SHA-256 (FIPS 180-4) over
//   parent digest (32 zero bytes for the first block) || B (u32) || the B tokens (i32)
//   || len(extra) (u32) || extra,  little-endian.
// Cached blocks whose count reaches zero wait in the free list (so the free-list order is
// the eviction order) and are revived from the middle of it on a hit; a block taken from
// the head for any use loses its digest.
//
// Each pool's free list is a doubly linked list over block ids (O(1) pop at the head,
// push at the tail and removal of a revived block).
#include <algorithm>
#include <atomic>
#include <condition_variable>
#include <cstdint>
#include <cstring>
#include <functional>
#include <mutex>
#include <new>
#include <string>
#include <thread>
#include <unordered_map>
#include <vector>

#include "../../include/pa.h"

namespace {

struct SeqState {
  std::vector<int32_t> table;  // block ids of the pool the sequence lives in
  int64_t ctx = 0;
  bool swapped = false;        // true: the ids are CPU-pool ids
};

// One pool of blocks: ordered free list (linked through prev/next) and reference counts.
struct Tier {
  int num_blocks = 0;
  std::vector<int32_t> prev, next;  // free-list links (-1 = none)
  std::vector<char> is_free;
  int32_t head = -1, tail = -1;
  int nfree = 0;
  std::vector<int32_t> refcount;

  bool init(int n, const int32_t* order) {
    num_blocks = n;
    prev.assign(n, -1);
    next.assign(n, -1);
    is_free.assign(n, 0);
    refcount.assign(n, 0);
    for (int i = 0; i < n; ++i) {
      const int32_t b = order ? order[i] : i;
      if (b < 0 || b >= n || is_free[b]) return false;
      push(b);
    }
    return true;
  }
  void push(int32_t b) {  // at the tail
    prev[b] = tail;
    next[b] = -1;
    if (tail >= 0) next[tail] = b; else head = b;
    tail = b;
    is_free[b] = 1;
    ++nfree;
  }
  void remove(int32_t b) {
    if (prev[b] >= 0) next[prev[b]] = next[b]; else head = next[b];
    if (next[b] >= 0) prev[next[b]] = prev[b]; else tail = prev[b];
    prev[b] = next[b] = -1;
    is_free[b] = 0;
    --nfree;
  }
  int32_t pop() {  // from the head; the caller has checked nfree
    const int32_t b = head;
    remove(b);
    refcount[b] = 1;
    return b;
  }
};

// ---- SHA-256 (FIPS 180-4) ----------------------------------------------------------
// The round constants are the first 32 bits of the fractional parts of the cube roots of
// the first 64 primes, the initial hash value those of the square roots of the first 8:
// computed here with exact integer roots rather than written out.
struct Sha256Consts {
  uint32_t k[64];
  uint32_t h0[8];
  Sha256Consts() {
    int primes[64];
    for (int n = 2, c = 0; c < 64; ++n) {
      bool prime = true;
      for (int d = 2; d * d <= n; ++d) prime = prime && n % d != 0;
      if (prime) primes[c++] = n;
    }
    for (int i = 0; i < 64; ++i) k[i] = static_cast<uint32_t>(iroot(primes[i], 3, 96));
    for (int i = 0; i < 8; ++i) h0[i] = static_cast<uint32_t>(iroot(primes[i], 2, 64));
  }
  // floor((p * 2^shift) ^ (1 / r)) by bisection on exact 128-bit integers; for r = 3 and
  // shift = 96 (r = 2, shift = 64) its low 32 bits are the fraction bits wanted.
  static unsigned __int128 iroot(int p, int r, int shift) {
    const unsigned __int128 target = static_cast<unsigned __int128>(p) << shift;
    unsigned __int128 lo = 0, hi = static_cast<unsigned __int128>(1) << (shift / r + 4);
    while (lo + 1 < hi) {
      const unsigned __int128 mid = (lo + hi) >> 1;
      unsigned __int128 pw = 1;
      for (int j = 0; j < r; ++j) pw *= mid;
      if (pw <= target) lo = mid; else hi = mid;
    }
    return lo;
  }
};

const Sha256Consts& sha_consts() {
  static const Sha256Consts c;
  return c;
}

inline uint32_t rotr(uint32_t x, int n) { return (x >> n) | (x << (32 - n)); }

class Sha256 {
 public:
  Sha256() { std::memcpy(h_, sha_consts().h0, sizeof(h_)); }
  void update(const uint8_t* p, size_t n) {
    bits_ += static_cast<uint64_t>(n) * 8;
    if (fill_ > 0) {  // top up a partly filled buffer
      const size_t take = n < static_cast<size_t>(64 - fill_) ? n : static_cast<size_t>(64 - fill_);
      std::memcpy(buf_ + fill_, p, take);
      fill_ += static_cast<int>(take);
      p += take;
      n -= take;
      if (fill_ < 64) return;
      block(buf_);
      fill_ = 0;
    }
    for (; n >= 64; p += 64, n -= 64) block(p);  // whole blocks straight from the input
    std::memcpy(buf_, p, n);
    fill_ = static_cast<int>(n);
  }
  void u32(uint32_t v) {
    uint8_t b[4] = {static_cast<uint8_t>(v), static_cast<uint8_t>(v >> 8),
                    static_cast<uint8_t>(v >> 16), static_cast<uint8_t>(v >> 24)};
    update(b, 4);
  }
  // Padding: a one bit, zeros up to 56 bytes into the last block (a further block when
  // fewer than 9 bytes are left), then the message length in bits, big-endian.
  void finish(uint8_t out[32]) {
    buf_[fill_++] = 0x80;
    if (fill_ > 56) {
      std::memset(buf_ + fill_, 0, static_cast<size_t>(64 - fill_));
      block(buf_);
      fill_ = 0;
    }
    std::memset(buf_ + fill_, 0, static_cast<size_t>(56 - fill_));
    for (int i = 0; i < 8; ++i) buf_[56 + i] = static_cast<uint8_t>(bits_ >> (56 - 8 * i));
    block(buf_);
    for (int i = 0; i < 8; ++i)
      for (int j = 0; j < 4; ++j) out[4 * i + j] = static_cast<uint8_t>(h_[i] >> (24 - 8 * j));
  }

 private:
  void block(const uint8_t* p) {
    const uint32_t* k = sha_consts().k;
    uint32_t w[64];
    for (int t = 0; t < 16; ++t)
      w[t] = (static_cast<uint32_t>(p[4 * t]) << 24) | (static_cast<uint32_t>(p[4 * t + 1]) << 16) |
             (static_cast<uint32_t>(p[4 * t + 2]) << 8) | p[4 * t + 3];
    for (int t = 16; t < 64; ++t) {
      const uint32_t s0 = rotr(w[t - 15], 7) ^ rotr(w[t - 15], 18) ^ (w[t - 15] >> 3);
      const uint32_t s1 = rotr(w[t - 2], 17) ^ rotr(w[t - 2], 19) ^ (w[t - 2] >> 10);
      w[t] = w[t - 16] + s0 + w[t - 7] + s1;
    }
    uint32_t a = h_[0], b = h_[1], c = h_[2], d = h_[3], e = h_[4], f = h_[5], g = h_[6],
             h = h_[7];
    for (int t = 0; t < 64; ++t) {
      const uint32_t t1 = h + (rotr(e, 6) ^ rotr(e, 11) ^ rotr(e, 25)) + ((e & f) ^ (~e & g)) +
                          k[t] + w[t];
      const uint32_t t2 = (rotr(a, 2) ^ rotr(a, 13) ^ rotr(a, 22)) + ((a & b) ^ (a & c) ^ (b & c));
      h = g;
      g = f;
      f = e;
      e = d + t1;
      d = c;
      c = b;
      b = a;
      a = t1 + t2;
    }
    h_[0] += a; h_[1] += b; h_[2] += c; h_[3] += d;
    h_[4] += e; h_[5] += f; h_[6] += g; h_[7] += h;
  }
  uint32_t h_[8];
  uint8_t buf_[64];
  int fill_ = 0;
  uint64_t bits_ = 0;
};

inline void put_u32(uint8_t* p, uint32_t v) {
  p[0] = static_cast<uint8_t>(v);
  p[1] = static_cast<uint8_t>(v >> 8);
  p[2] = static_cast<uint8_t>(v >> 16);
  p[3] = static_cast<uint8_t>(v >> 24);
}

// A 32-byte digest held by value (no allocation).
struct Digest {
  uint64_t w[4];
  bool operator==(const Digest& o) const {
    return w[0] == o.w[0] && w[1] == o.w[1] && w[2] == o.w[2] && w[3] == o.w[3];
  }
};

// The digests that name device blocks, and the lookup from a digest to its block: an
// open-addressing table (linear probing; a removal shifts the entries after it back, so
// no deleted markers build up).  A slot holds a block id and the low 32 bits of the
// block's digest (SHA-256 output is uniformly distributed: those bits pick the home slot
// and reject most mismatches without reading the digest).  A block carries at most one
// digest, so with at least twice as many slots as blocks the table is at most half full
// and every probe meets an empty slot.  Nothing is allocated after init.
class DigestTable {
 public:
  void init(int num_blocks) {
    size_t cap = 16;
    while (cap < 2 * static_cast<size_t>(num_blocks)) cap <<= 1;
    slot_.assign(cap, Slot{-1, 0});
    mask_ = static_cast<uint32_t>(cap - 1);
    key_.assign(static_cast<size_t>(num_blocks), Digest{});
    named_.assign(static_cast<size_t>(num_blocks), 0);
    size_ = 0;
  }
  // the block named d, or -1
  int32_t find(const Digest& d) const {
    const uint32_t tag = tag_of(d);
    for (uint32_t i = tag & mask_;; i = (i + 1) & mask_) {
      const Slot& e = slot_[i];
      if (e.block < 0) return -1;
      if (e.tag == tag && key_[e.block] == d) return e.block;
    }
  }
  bool named(int32_t b) const { return named_[b] != 0; }
  const Digest& digest(int32_t b) const { return key_[b]; }
  // name block b (unnamed) by d (naming no block)
  void name(int32_t b, const Digest& d) {
    key_[b] = d;
    named_[b] = 1;
    const uint32_t tag = tag_of(d);
    uint32_t i = tag & mask_;
    while (slot_[i].block >= 0) i = (i + 1) & mask_;
    slot_[i] = Slot{b, tag};
    ++size_;
  }
  // take block b's (present) digest away
  void unname(int32_t b) {
    uint32_t i = tag_of(key_[b]) & mask_;
    while (slot_[i].block != b) i = (i + 1) & mask_;
    // Close the hole at i: an entry further along the run moves into it when the hole
    // lies on that entry's probe path (between its home slot and where it sits).
    for (uint32_t j = (i + 1) & mask_; slot_[j].block >= 0; j = (j + 1) & mask_) {
      const uint32_t h = slot_[j].tag & mask_;
      if (((j - h) & mask_) >= ((j - i) & mask_)) {
        slot_[i] = slot_[j];
        i = j;
      }
    }
    slot_[i] = Slot{-1, 0};
    named_[b] = 0;
    --size_;
  }
  int size() const { return size_; }

 private:
  struct Slot {
    int32_t block;  // -1: empty
    uint32_t tag;   // low 32 bits of the block's digest
  };
  static uint32_t tag_of(const Digest& d) { return static_cast<uint32_t>(d.w[0]); }
  std::vector<Slot> slot_;
  uint32_t mask_ = 0;
  std::vector<Digest> key_;
  std::vector<char> named_;
  int size_ = 0;
};

// Digests of the n / B full blocks of a token list, chained.  Each block's message is
// laid out in one buffer and hashed in one pass.
std::vector<Digest> block_digests(const int32_t* tokens, int n, int bs, const uint8_t* extra,
                                  int extra_len) {
  std::vector<Digest> out;
  const int m = n / bs;
  out.reserve(static_cast<size_t>(m));
  std::vector<uint8_t> msg(32 + 4 + 4 * static_cast<size_t>(bs) + 4);
  uint8_t parent[32] = {0};
  for (int i = 0; i < m; ++i) {
    std::memcpy(msg.data(), parent, 32);
    put_u32(msg.data() + 32, static_cast<uint32_t>(bs));
    for (int j = 0; j < bs; ++j)
      put_u32(msg.data() + 36 + 4 * j, static_cast<uint32_t>(tokens[i * bs + j]));
    put_u32(msg.data() + 36 + 4 * bs, static_cast<uint32_t>(extra_len));
    Sha256 h;
    h.update(msg.data(), msg.size());
    if (extra_len > 0) h.update(extra, static_cast<size_t>(extra_len));
    h.finish(parent);
    Digest d;
    std::memcpy(d.w, parent, 32);
    out.push_back(d);
  }
  return out;
}

// A small persistent pool of host threads for the per-request digest chains of a batch
// (independent across requests).  Created on first use; the calling thread works too.
class Workers {
 public:
  static Workers& get() {
    static Workers* w = new Workers();  // never destroyed: its threads live with the process
    return *w;
  }
  int size() const { return static_cast<int>(threads_.size()) + 1; }
  // fn(i) for i in [0, total), spread over the pool; returns when every call is done.
  void run(int total, const std::function<void(int)>& fn) {
    std::lock_guard<std::mutex> one_at_a_time(run_m_);
    if (threads_.empty() || total <= 1) {
      for (int i = 0; i < total; ++i) fn(i);
      return;
    }
    std::unique_lock<std::mutex> lk(m_);
    job_ = &fn;
    total_ = total;
    next_.store(0);
    busy_ = static_cast<int>(threads_.size());
    ++gen_;
    cv_.notify_all();
    lk.unlock();
    work();
    lk.lock();
    done_.wait(lk, [&] { return busy_ == 0; });
    job_ = nullptr;
  }

 private:
  Workers() {
    unsigned hw = std::thread::hardware_concurrency();
    int n = hw > 1 ? static_cast<int>(hw > 16 ? 16 : hw) - 1 : 0;
    for (int i = 0; i < n; ++i) threads_.emplace_back([this] { loop(); });
    for (std::thread& t : threads_) t.detach();
  }
  void work() {
    for (int i; (i = next_.fetch_add(1)) < total_;) (*job_)(i);
  }
  void loop() {
    uint64_t seen = 0;
    for (;;) {
      std::unique_lock<std::mutex> lk(m_);
      cv_.wait(lk, [&] { return gen_ != seen; });
      seen = gen_;
      lk.unlock();
      work();
      lk.lock();
      if (--busy_ == 0) done_.notify_one();
    }
  }
  std::vector<std::thread> threads_;
  std::mutex run_m_, m_;
  std::condition_variable cv_, done_;
  const std::function<void(int)>* job_ = nullptr;
  int total_ = 0;
  std::atomic<int> next_{0};
  int busy_ = 0;
  uint64_t gen_ = 0;
};

}  // namespace

struct pa_pool {
  int block_size = 0;
  Tier gpu, cpu;
  std::unordered_map<int64_t, SeqState> seqs;
  DigestTable names;  // digests of cached device blocks, and digest -> block

  // a device block from the head of the free list; a cached one is evicted
  int32_t take() {
    const int32_t b = gpu.pop();
    if (names.named(b)) names.unname(b);
    return b;
  }
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
    p->names.init(num_blocks);
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
  for (int64_t i = 0; i < need; ++i) st.table.push_back(pool->take());
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
    st.table.push_back(pool->take());
  } else if (g.refcount[st.table.back()] > 1) {
    // The partly filled last block is shared: copy it before writing.
    if (g.nfree < 1) return PA_ERR_POOL_EXHAUSTED;
    if (!cow_src || !cow_dst) return PA_ERR_ARG;
    int32_t old_b = st.table.back();
    int32_t new_b = pool->take();
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
    moved[i] = to_cpu ? dst.pop() : pool->take();
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
  int i = 0;
  for (int32_t b = t.head; b >= 0 && i < cap; b = t.next[b]) out[i++] = b;
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

// Prefill with prefix caching of one request whose digests are known.
static int allocate_prefix_core(pa_pool* pool, int64_t seq_id, int n_tokens,
                                const std::vector<Digest>& dg, int* cached_tokens_out) {
  if (pool->seqs.count(seq_id)) return PA_ERR_UNKNOWN_SEQ;
  const int bs = pool->block_size;
  // the longest run of leading full blocks already cached
  std::vector<int32_t> hits;
  for (const Digest& d : dg) {
    const int32_t b = pool->names.find(d);
    if (b < 0) break;
    hits.push_back(b);
  }
  const int64_t nblk = (static_cast<int64_t>(n_tokens) + bs - 1) / bs;
  const int64_t need = nblk - static_cast<int64_t>(hits.size());
  int64_t revived = 0;
  for (int32_t b : hits) revived += pool->gpu.refcount[b] == 0;
  if (need > pool->gpu.nfree - revived) return PA_ERR_POOL_EXHAUSTED;
  SeqState st;
  st.table.reserve(static_cast<size_t>(nblk) + 1);
  for (int32_t b : hits) {
    if (pool->gpu.refcount[b] == 0) pool->gpu.remove(b);
    pool->gpu.refcount[b] += 1;
    st.table.push_back(b);
  }
  for (int64_t i = 0; i < need; ++i) st.table.push_back(pool->take());
  for (size_t i = hits.size(); i < dg.size(); ++i) {
    if (pool->names.find(dg[i]) >= 0) continue;  // another block answers it
    pool->names.name(st.table[i], dg[i]);
  }
  st.ctx = n_tokens;
  pool->seqs.emplace(seq_id, std::move(st));
  if (cached_tokens_out) *cached_tokens_out = static_cast<int>(hits.size()) * bs;
  return PA_OK;
}

// Lookups and allocation of a batch whose digests are known, in request order, with the
// slots of the uncached tokens and the block tables written out.
static int place_batch(pa_pool* pool, int n, const int64_t* seq_ids, const std::vector<int>& lens,
                       const std::vector<std::vector<Digest>>& dg, int* cached_out,
                       int64_t* slots_out, int32_t* tables_out, int table_width, int* n_done) {
  const int bs = pool->block_size;
  int64_t o = 0;
  for (int r = 0; r < n; ++r) {
    const int len = lens[r];
    int cached = 0;
    const int st = allocate_prefix_core(pool, seq_ids[r], len, dg[r], &cached);
    if (st < 0) return st;
    cached_out[r] = cached;
    const SeqState& seq = pool->seqs.find(seq_ids[r])->second;
    if (slots_out)  // block by block: slot = block * B + offset, no division per token
      for (int t = cached; t < len;) {
        const int64_t base = static_cast<int64_t>(seq.table[t / bs]) * bs;
        const int end = std::min(len, (t / bs + 1) * bs);
        for (int off = t % bs; t < end; ++t, ++off) slots_out[o++] = base + off;
      }
    if (tables_out) {
      int32_t* row = tables_out + static_cast<size_t>(r) * table_width;
      const int nt = static_cast<int>(seq.table.size());
      for (int j = 0; j < table_width; ++j) row[j] = j < nt ? seq.table[j] : 0;
    }
    if (n_done) *n_done = r + 1;
  }
  return PA_OK;
}

extern "C" {

int pa_pool_allocate_prefix(pa_pool* pool, int64_t seq_id, const int32_t* tokens, int n_tokens,
                            const uint8_t* extra, int extra_len, int* cached_tokens_out) {
  if (!pool || n_tokens < 0 || (n_tokens > 0 && !tokens) || extra_len < 0 ||
      (extra_len > 0 && !extra))
    return PA_ERR_ARG;
  if (pool->seqs.count(seq_id)) return PA_ERR_UNKNOWN_SEQ;
  std::vector<Digest> dg;
  try {
    dg = block_digests(tokens, n_tokens, pool->block_size, extra, extra_len);
    return allocate_prefix_core(pool, seq_id, n_tokens, dg, cached_tokens_out);
  } catch (...) {
    return PA_ERR_ARG;
  }
}

int pa_pool_table_width(const pa_pool* pool, int n, const int64_t* token_start) {
  if (!pool || n < 0 || (n > 0 && !token_start)) return PA_ERR_ARG;
  if (n > 0 && token_start[0] < 0) return PA_ERR_ARG;
  const int64_t bs = pool->block_size;
  int64_t width = 0;
  for (int r = 0; r < n; ++r) {
    const int64_t len = token_start[r + 1] - token_start[r];
    if (len < 0 || len > 0x7fffffff) return PA_ERR_ARG;
    width = std::max(width, (len + bs - 1) / bs);
  }
  return static_cast<int>(width);
}

int pa_pool_allocate_prefix_batch(pa_pool* pool, int n, const int64_t* seq_ids,
                                  const int32_t* tokens, const int64_t* token_start,
                                  const uint8_t* extras, const int64_t* extra_start,
                                  int* cached_out, int64_t* slots_out, int32_t* tables_out,
                                  int table_width, int* n_done) {
  if (n_done) *n_done = 0;
  if (!pool || n < 0 || (n > 0 && (!seq_ids || !token_start || !cached_out)) || table_width < 0 ||
      (extras && !extra_start))
    return PA_ERR_ARG;
  if (n == 0) return PA_OK;
  const int bs = pool->block_size;
  if (token_start[0] < 0 || (extras && extra_start[0] < 0)) return PA_ERR_ARG;
  for (int r = 0; r < n; ++r) {
    const int64_t len = token_start[r + 1] - token_start[r];
    if (len < 0 || len > 0x7fffffff || (len > 0 && !tokens)) return PA_ERR_ARG;
    if (extras && (extra_start[r + 1] < extra_start[r] ||
                   extra_start[r + 1] - extra_start[r] > 0x7fffffff))
      return PA_ERR_ARG;
    if (tables_out && (len + bs - 1) / bs > table_width) return PA_ERR_ARG;
  }
  try {
    // the digest chains, one request per task
    std::vector<std::vector<Digest>> dg(static_cast<size_t>(n));
    std::atomic<bool> failed{false};
    const std::function<void(int)> hash_one = [&](int r) {
      try {
        const int64_t a = token_start[r];
        const int len = static_cast<int>(token_start[r + 1] - a);
        const uint8_t* ex = extras ? extras + extra_start[r] : nullptr;
        const int ex_len = extras ? static_cast<int>(extra_start[r + 1] - extra_start[r]) : 0;
        dg[r] = block_digests(tokens + a, len, bs, ex, ex_len);
      } catch (...) {
        failed.store(true);
      }
    };
    int64_t total_blocks = (token_start[n] - token_start[0]) / bs;
    if (total_blocks >= 256)
      Workers::get().run(n, hash_one);
    else
      for (int r = 0; r < n; ++r) hash_one(r);
    if (failed.load()) return PA_ERR_ARG;
    std::vector<int> lens(static_cast<size_t>(n));
    for (int r = 0; r < n; ++r) lens[r] = static_cast<int>(token_start[r + 1] - token_start[r]);
    return place_batch(pool, n, seq_ids, lens, dg, cached_out, slots_out, tables_out, table_width,
                       n_done);
  } catch (...) {
    return PA_ERR_ARG;
  }
}

int pa_pool_allocate_hashed_batch(pa_pool* pool, int n, const int64_t* seq_ids,
                                  const int32_t* n_tokens, const uint8_t* digests,
                                  int* cached_out, int64_t* slots_out, int32_t* tables_out,
                                  int table_width, int* n_done) {
  if (n_done) *n_done = 0;
  if (!pool || n < 0 || (n > 0 && (!seq_ids || !n_tokens || !cached_out)) || table_width < 0)
    return PA_ERR_ARG;
  if (n == 0) return PA_OK;
  const int bs = pool->block_size;
  try {
    std::vector<int> lens(static_cast<size_t>(n));
    std::vector<std::vector<Digest>> dg(static_cast<size_t>(n));
    const uint8_t* d = digests;
    for (int r = 0; r < n; ++r) {
      lens[r] = n_tokens[r];
      if (lens[r] < 0 ||
          (tables_out && (static_cast<int64_t>(lens[r]) + bs - 1) / bs > table_width))
        return PA_ERR_ARG;
      const int m = lens[r] / bs;
      if (m > 0 && !digests) return PA_ERR_ARG;
      dg[r].resize(static_cast<size_t>(m));
      for (int i = 0; i < m; ++i, d += 32) std::memcpy(dg[r][i].w, d, 32);
    }
    return place_batch(pool, n, seq_ids, lens, dg, cached_out, slots_out, tables_out, table_width,
                       n_done);
  } catch (...) {
    return PA_ERR_ARG;
  }
}

int pa_pool_free_batch(pa_pool* pool, const int64_t* seq_ids, int n) {
  if (!pool || n < 0 || (n > 0 && !seq_ids)) return PA_ERR_ARG;
  for (int r = 0; r < n; ++r) {
    const int st = pa_pool_free(pool, seq_ids[r]);
    if (st < 0) return st;
  }
  return PA_OK;
}

int pa_pool_num_cached(const pa_pool* pool) {
  return pool ? pool->names.size() : PA_ERR_ARG;
}

int pa_pool_block_digest(const pa_pool* pool, int32_t block, uint8_t* digest_out) {
  if (!pool || !digest_out || block < 0 || block >= pool->gpu.num_blocks) return PA_ERR_ARG;
  if (!pool->names.named(block)) return 0;
  std::memcpy(digest_out, pool->names.digest(block).w, 32);
  return 1;
}

int pa_prefix_block_hashes(const int32_t* tokens, int n_tokens, int block_size,
                           const uint8_t* extra, int extra_len, uint8_t* digests_out, int cap) {
  if (n_tokens < 0 || (n_tokens > 0 && !tokens) || block_size <= 0 || extra_len < 0 ||
      (extra_len > 0 && !extra) || cap < 0)
    return PA_ERR_ARG;
  const int m = n_tokens / block_size;
  if (m > cap || (m > 0 && !digests_out)) return PA_ERR_ARG;
  const std::vector<Digest> dg = block_digests(tokens, n_tokens, block_size, extra, extra_len);
  for (int i = 0; i < m; ++i) std::memcpy(digests_out + 32 * i, dg[i].w, 32);
  return m;
}

int pa_sha256(const void* data, size_t len, uint8_t* digest_out) {
  if ((len > 0 && !data) || !digest_out) return PA_ERR_ARG;
  Sha256 h;
  h.update(static_cast<const uint8_t*>(data), len);
  h.finish(digest_out);
  return PA_OK;
}

}  // extern "C"
