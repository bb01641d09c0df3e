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

Readings where the pages are silent:
* a write copies when the last block's reference count is above one at write time, so
  with k sharers the first k-1 writers copy and the last writes in place;
* blocks freed together return to the tail in table order;
* an operation that cannot get every block it needs changes nothing.
"""
import math


class PoolExhausted(Exception):
    """Not enough free blocks; the pool is unchanged."""


class UnknownSequence(KeyError):
    """The sequence id is not live (or, for allocate/fork targets, already live)."""


class BlockPool:
    def __init__(self, num_blocks, block_size, initial_free_order=None):
        if initial_free_order is None:
            initial_free_order = range(num_blocks)
        order = [int(b) for b in initial_free_order]
        if sorted(order) != list(range(num_blocks)):
            raise ValueError("initial free order must be a permutation of 0..num_blocks-1")
        self.num_blocks = num_blocks
        self.block_size = block_size
        self.free_list = order          # head = index 0
        self.refcount = [0] * num_blocks
        self.tables = {}                # seq id -> list of physical block ids
        self.ctx = {}                   # seq id -> tokens held

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
        return blocks

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
        self.tables[child] = list(self.tables[parent])
        self.ctx[child] = self.ctx[parent]
        for b in self.tables[child]:
            self.refcount[b] += 1

    def free(self, seq):
        """End a sequence: drop one reference per block; blocks at zero go to the tail."""
        if seq not in self.tables:
            raise UnknownSequence(seq)
        for b in self.tables.pop(seq):
            self.refcount[b] -= 1
            if self.refcount[b] == 0:
                self.free_list.append(b)
        del self.ctx[seq]
