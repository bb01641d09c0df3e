"""Host block bookkeeping: free list, reference counts, fork, copy-on-write.

Test infrastructure only.  The steps, in the pages' order:

* Physical blocks of B tokens sit in a free pool.  A sequence takes a block from the pool
  each time it grows by B tokens and returns all its blocks when it ends
  (daiw.org "Paged Attention", section 定义, 分配).
* Prefill takes ceil(prompt / B) blocks; decode adds one block every B tokens; a finished
  sequence returns every block (horeb.top, section 分配策略).
* The free pool is an ordered list: blocks are taken from its head and returned to its
  tail (aiqz.cc "vLLM PagedAttention engine", section Python 演示 -- the demo allocator
  slices the first n free blocks, pops index 0 on growth and appends freed blocks).
* A physical block may be referenced by several sequences and is reclaimed only when its
  reference count reaches zero (daiw.org, section 量化, Copy-on-write / 共享).
* Fork: a new sequence shares its parent's block chain (daiw.org, section 工程现场,
  Copy-on-write 与 fork; chenyuan1125, section 一块内存…).
* Copy-on-write: when a branch must write into a last block that is still shared, the
  block is copied, that branch's mapping is updated and the write proceeds; full old
  blocks stay shared (chenyuan1125, section 一块内存…; horeb.top, section 内存共享).
* When the pool is exhausted the request is rejected rather than the process failing
  (daiw.org, section 速查卡, 运维提示; the demo's allocate returns False).
* Automatic prefix caching: a full block is identified by its parent block's hash, its
  own tokens and extra keys (LoRA, multimodal inputs, a cache salt), so that a new
  request whose prompt starts with the same blocks finds and reuses their K/V instead of
  recomputing them (chenyuan1125 "vllm-pagedattention", section 一块内存，如何安全地属于
  多条序列); which cached blocks to keep is an eviction policy, and a per-tenant salt
  keeps tenants' prefixes apart (same page, section 分页不是免费午餐).
* Preemption: when device memory runs short, a request's blocks can be moved out whole
  into CPU memory and moved back once room returns; the block table is what makes the
  move cheap (aiqz.cc, section 连续批处理：随到随走的新秩序).  The CPU side is a second
  pool of blocks with the same free list and reference count rules.

Readings where the pages are silent:
* a write copies when the last block's reference count is above one at write time, so
  with k sharers the first k-1 writers copy and the last writes in place;
* blocks freed together return to the tail in table order;
* an operation that cannot get every block it needs changes nothing;
* swap_out moves a group of resident sequences: every distinct device block of their
  tables (sequences in the order given, tables in order, first appearance) gets one CPU
  block from the head of the CPU free list, carrying the group's references; the device
  block loses those references and, at zero, returns to the device tail in that same
  order.  swap_in is the mirror image.  A block also held outside the group keeps its
  other references where it is (the group then owns a separate copy);
* a swapped-out sequence can be freed (its CPU blocks return to the CPU tail) or swapped
  in, but not grown or forked;
* prefix hashing: digest_i = SHA-256(digest_{i-1} || B as u32 || the block's B tokens as
  i32 || len(extra) as u32 || extra), all little-endian, digest_{-1} = 32 zero bytes;
  the request's extra bytes (salt, adapter id, ...) enter every block;
* a prompt's lookup walks its full blocks in order and stops at the first miss; a hit
  adds a reference (a cached block sitting in the free list leaves it); the rest of the
  prompt gets fresh blocks from the head, and every full block among them is registered
  under its digest unless that digest already names a block;
* a cached block whose count reaches zero stays cached in the free list (eviction order =
  free-list order); it is evicted -- its digest forgotten -- when it is taken from the
  head for any other use.  Partly filled blocks and blocks filled by decode are not
  registered.
"""
import hashlib
import math
import struct


class PoolExhausted(Exception):
    """Not enough free blocks; the pool is unchanged."""


class UnknownSequence(KeyError):
    """The sequence id is not live (or, for allocate/fork targets, already live)."""


class WrongTier(Exception):
    """The sequence is swapped out where a resident one is needed, or the reverse."""


def block_hashes(tokens, block_size, extra=b""):
    """Chained SHA-256 digests of the full blocks of a token list (hashlib)."""
    tokens = [int(t) for t in tokens]
    extra = bytes(extra)
    out, parent = [], bytes(32)
    for i in range(len(tokens) // block_size):
        blk = tokens[i * block_size:(i + 1) * block_size]
        msg = (parent + struct.pack("<I", block_size) + struct.pack(f"<{block_size}i", *blk)
               + struct.pack("<I", len(extra)) + extra)
        parent = hashlib.sha256(msg).digest()
        out.append(parent)
    return out


def _order(n, order):
    order = list(range(n)) if order is None else [int(b) for b in order]
    if sorted(order) != list(range(n)):
        raise ValueError("a free order must be a permutation of 0..n-1")
    return order


class BlockPool:
    def __init__(self, num_blocks, block_size, initial_free_order=None, num_cpu_blocks=0,
                 cpu_free_order=None):
        self.num_blocks = num_blocks
        self.block_size = block_size
        self.free_list = _order(num_blocks, initial_free_order)   # head = index 0
        self.refcount = [0] * num_blocks
        self.num_cpu_blocks = num_cpu_blocks
        self.cpu_free_list = _order(num_cpu_blocks, cpu_free_order)
        self.cpu_refcount = [0] * num_cpu_blocks
        self.tables = {}                # seq id -> list of block ids (CPU ids if swapped)
        self.ctx = {}                   # seq id -> tokens held
        self.swapped = set()            # seq ids whose blocks are in the CPU pool
        self.digest_of = [None] * num_blocks   # device block -> its registered digest
        self.cached = {}                # digest -> device block

    # -- queries ------------------------------------------------------------------------
    def num_free(self):
        return len(self.free_list)

    def block_table(self, seq):
        if seq not in self.tables:
            raise UnknownSequence(seq)
        return list(self.tables[seq])

    def context_len(self, seq):
        if seq not in self.ctx:
            raise UnknownSequence(seq)
        return self.ctx[seq]

    def is_swapped(self, seq):
        if seq not in self.tables:
            raise UnknownSequence(seq)
        return seq in self.swapped

    def slot(self, seq, t):
        """Slot of logical token t of ``seq``: table[t // B] * B + t % B."""
        table = self.tables[seq]
        return table[t // self.block_size] * self.block_size + t % self.block_size

    # -- operations ---------------------------------------------------------------------
    def _take(self, n):
        if n > len(self.free_list):
            raise PoolExhausted(f"need {n} blocks, {len(self.free_list)} free")
        blocks = self.free_list[:n]
        del self.free_list[:n]
        for b in blocks:
            self.refcount[b] = 1
            self._evict(b)
        return blocks

    def _evict(self, b):
        if self.digest_of[b] is not None:
            del self.cached[self.digest_of[b]]
            self.digest_of[b] = None

    def num_cached(self):
        return len(self.cached)

    def allocate_prefix(self, seq, tokens, extra=b""):
        """Prefill with prefix caching: reuse the cached blocks of the longest run of
        leading full blocks, take fresh blocks for the rest, register the new full blocks.
        Returns the number of leading tokens whose K/V are already cached."""
        if seq in self.tables:
            raise UnknownSequence(f"sequence {seq} already live")
        n = len(tokens)
        digests = block_hashes(tokens, self.block_size, extra)
        hits = []
        for dg in digests:
            if dg not in self.cached:
                break
            hits.append(self.cached[dg])
        need = math.ceil(n / self.block_size) - len(hits)
        revived = sum(1 for b in hits if self.refcount[b] == 0)
        if need > len(self.free_list) - revived:
            raise PoolExhausted(f"need {need} blocks, {len(self.free_list) - revived} free")
        for b in hits:
            if self.refcount[b] == 0:
                self.free_list.remove(b)
            self.refcount[b] += 1
        fresh = self._take(need)
        table = hits + fresh
        for i in range(len(hits), len(digests)):
            if digests[i] not in self.cached:
                self.cached[digests[i]] = table[i]
                self.digest_of[table[i]] = digests[i]
        self.tables[seq] = table
        self.ctx[seq] = n
        return len(hits) * self.block_size

    def allocate(self, seq, n_tokens):
        """Prefill: give a new sequence ceil(n_tokens / B) blocks holding n_tokens tokens."""
        if seq in self.tables:
            raise UnknownSequence(f"sequence {seq} already live")
        if n_tokens < 0:
            raise ValueError("n_tokens < 0")
        self.tables[seq] = self._take(math.ceil(n_tokens / self.block_size))
        self.ctx[seq] = n_tokens

    def append_slot(self, seq):
        """Reserve the slot of the sequence's next token.

        Returns (slot, cow) where cow is None or the (src, dst) block pair the caller must
        copy before writing.  A new block is taken when the last one is full; a shared,
        partly filled last block is copied first.
        """
        if seq not in self.tables:
            raise UnknownSequence(seq)
        if seq in self.swapped:
            raise WrongTier(f"sequence {seq} is swapped out")
        table = self.tables[seq]
        t = self.ctx[seq]
        cow = None
        if t % self.block_size == 0:
            table.extend(self._take(1))
        elif self.refcount[table[-1]] > 1:
            old = table[-1]
            (new,) = self._take(1)
            self.refcount[old] -= 1
            table[-1] = new
            cow = (old, new)
        self.ctx[seq] = t + 1
        return self.slot(seq, t), cow

    def fork(self, parent, child):
        """The child shares every block of the parent's chain (reference counts + 1)."""
        if parent not in self.tables:
            raise UnknownSequence(parent)
        if child in self.tables:
            raise UnknownSequence(f"sequence {child} already live")
        if parent in self.swapped:
            raise WrongTier(f"sequence {parent} is swapped out")
        self.tables[child] = list(self.tables[parent])
        self.ctx[child] = self.ctx[parent]
        for b in self.tables[child]:
            self.refcount[b] += 1

    def free(self, seq):
        """End a sequence: drop one reference per block; blocks at zero go to the tail."""
        if seq not in self.tables:
            raise UnknownSequence(seq)
        on_cpu = seq in self.swapped
        refcount = self.cpu_refcount if on_cpu else self.refcount
        free_list = self.cpu_free_list if on_cpu else self.free_list
        for b in self.tables.pop(seq):
            refcount[b] -= 1
            if refcount[b] == 0:
                free_list.append(b)
        del self.ctx[seq]
        self.swapped.discard(seq)

    def _move(self, seqs, to_cpu):
        """Move a group of sequences to the other pool; return the (from, to) block pairs
        the caller copies."""
        seqs = list(seqs)
        if len(set(seqs)) != len(seqs):
            raise ValueError("a sequence appears twice in the group")
        for seq in seqs:
            if seq not in self.tables:
                raise UnknownSequence(seq)
            if (seq in self.swapped) == to_cpu:
                raise WrongTier(f"sequence {seq} is already {'out' if to_cpu else 'in'}")
        src_ref, src_free = ((self.refcount, self.free_list) if to_cpu
                             else (self.cpu_refcount, self.cpu_free_list))
        dst_ref, dst_free = ((self.cpu_refcount, self.cpu_free_list) if to_cpu
                             else (self.refcount, self.free_list))
        # the group's references to each distinct block, in order of first appearance
        refs = {}
        for seq in seqs:
            for b in self.tables[seq]:
                refs[b] = refs.get(b, 0) + 1
        if len(refs) > len(dst_free):
            raise PoolExhausted(f"need {len(refs)} blocks, {len(dst_free)} free")
        new = dict(zip(refs, dst_free[:len(refs)]))
        del dst_free[:len(refs)]
        if not to_cpu:
            for b in new.values():
                self._evict(b)
        for b, n in refs.items():
            dst_ref[new[b]] = n
            src_ref[b] -= n
            if src_ref[b] == 0:
                src_free.append(b)
        for seq in seqs:
            self.tables[seq] = [new[b] for b in self.tables[seq]]
            if to_cpu:
                self.swapped.add(seq)
            else:
                self.swapped.discard(seq)
        return [(b, new[b]) for b in refs]

    def swap_out(self, seqs):
        """Preempt a group of resident sequences: returns (device block, CPU block) pairs."""
        return self._move(seqs, True)

    def swap_in(self, seqs):
        """Bring a group of swapped-out sequences back: returns (CPU block, device block)
        pairs."""
        return self._move(seqs, False)
