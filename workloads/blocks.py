"""Host-side block bookkeeping used to build workloads: a free list popped in a
seeded order, per-block reference counts, sharing and copy-on-write.

This is input generation.  It decides which physical block each logical block
of a sequence occupies and which blocks must be copied before a write; it never
computes flat slot numbers, never touches K/V values and holds none of the
attention arithmetic.

Behaviour follows "vLLM Framework and Inference Engine Design", section "How is
vLLM's KV cache paged?" (bullets "Growing", "Sharing", "Freeing"): a full last
block is followed by a block popped from the free list in constant time; every
block carries a reference count; and, from section "What operations can cause
memory fragmentation ...", a shared block is copied only when a sequence needs
to write into it (copy-on-write).
"""
from collections import deque


class BlockPool:
    """Free list of physical block ids plus reference counts."""

    def __init__(self, num_blocks, free_order):
        free_order = [int(b) for b in free_order]
        if sorted(free_order) != list(range(num_blocks)):
            raise ValueError("free_order must be a permutation of range(num_blocks)")
        self.num_blocks = num_blocks
        self.free = deque(free_order)
        self.ref = [0] * num_blocks

    def allocate(self):
        if not self.free:
            raise MemoryError("block pool exhausted")
        b = self.free.popleft()
        self.ref[b] = 1
        return b

    def share(self, b):
        self.ref[b] += 1

    def release(self, b):
        if self.ref[b] <= 0:
            raise ValueError("release of a free block %d" % b)
        self.ref[b] -= 1
        if self.ref[b] == 0:
            self.free.append(b)

    def num_free(self):
        return len(self.free)


class Sequence:
    """A sequence's block table and token count."""

    def __init__(self, pool, block_size):
        self.pool = pool
        self.B = block_size
        self.table = []
        self.num_tokens = 0

    def fork(self):
        """A new sequence sharing every block of this one (refcounts + 1)."""
        child = Sequence(self.pool, self.B)
        child.table = list(self.table)
        child.num_tokens = self.num_tokens
        for b in self.table:
            self.pool.share(b)
        return child

    def reserve(self, n):
        """Grow to hold n more tokens.  Returns the copy-on-write (src, dst)
        pairs needed before those tokens are written: a shared, partially
        filled last block is replaced by a private copy."""
        copies = []
        if n <= 0:
            return copies
        filled_in_last = self.num_tokens - (len(self.table) - 1) * self.B if self.table else 0
        if self.table and filled_in_last < self.B and self.pool.ref[self.table[-1]] > 1:
            src = self.table[-1]
            dst = self.pool.allocate()
            self.pool.release(src)
            self.table[-1] = dst
            copies.append((src, dst))
        target = self.num_tokens + n
        while len(self.table) * self.B < target:
            self.table.append(self.pool.allocate())
        self.num_tokens = target
        return copies

    def release_before_window(self, W):
        """Sliding-window attention ("How does it support prompts of arbitrary
        length? Does it have a sliding window?"): with each token attending
        only to the last W, blocks wholly before the window are released; their
        table entries become -1 (logical indices stay as they are)."""
        first = max(0, self.num_tokens - W) // self.B   # first block still in the window
        for j in range(min(first, len(self.table))):
            if self.table[j] >= 0:
                self.pool.release(self.table[j])
                self.table[j] = -1

    def release(self):
        for b in self.table:
            if b >= 0:
                self.pool.release(b)
        self.table = []
        self.num_tokens = 0
