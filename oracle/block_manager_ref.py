"""Reference block manager: free list, refcounts, on-demand allocation, fork,
copy-on-write.  Pure bookkeeping, one token at a time.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

Follows the BlockManager sketch of "How LLM Inference Engines Work ..."
(letsbuildsolutions.com, section "PagedAttention: Virtual Memory for KV
Caches"): a free list used as a stack (allocation pops the end, freeing
pushes back), a new block starts with refcount 1 and is appended to the
sequence's logical block list, allocation fails (returns False) on an empty
free list, and freeing a sequence decrements each of its blocks and returns
a block to the free list when its count reaches zero.

Added from the other pages, with the readings taken:
  * On-demand allocation (ontq section 3): a block is taken only when the
    previous one is full, i.e. just before writing token t with t % B == 0.
  * Sharing and copy-on-write (ontq section 3; thewebvale section 2): a
    forked sequence points at its parent's blocks (each refcount + 1).  When
    a sequence writes into a block whose refcount is above 1, it takes a
    fresh block, queues a copy (old -> new) of the whole block, drops one
    reference to the old block, and writes into the new one.  A sequence
    that finds refcount 1 writes in place.  Within one call sequences are
    served in the order given.
  * A multi-token request either succeeds as a whole or changes nothing.
  * Slot of token t: table[t // B] * B + t % B (thewebvale section 2).
  * The initial free list order is given by the caller.
"""

from __future__ import annotations

import copy


class RefBlockManager:
    def __init__(self, block_size: int, free_order):
        self.B = int(block_size)
        self.num_blocks = len(free_order)
        self.free = [int(b) for b in free_order]
        self.refcount = {}
        self.blocks = {}
        self.length = {}
        self.copies = []

    # -- the sketch's two operations -------------------------------------
    def _allocate(self, seq) -> bool:
        if len(self.free) == 0:
            return False
        blk = self.free.pop()
        self.refcount[blk] = 1
        self.blocks[seq].append(blk)
        return True

    def free_seq(self, seq) -> None:
        for blk in self.blocks[seq]:
            self.refcount[blk] -= 1
            if self.refcount[blk] == 0:
                self.free.append(blk)
                del self.refcount[blk]
        del self.blocks[seq]
        del self.length[seq]

    # -- sharing ---------------------------------------------------------
    def fork(self, parent, child) -> None:
        self.blocks[child] = list(self.blocks[parent])
        self.length[child] = self.length[parent]
        for blk in self.blocks[child]:
            self.refcount[blk] += 1

    # -- writing tokens --------------------------------------------------
    def _append_one(self, seq):
        t = self.length[seq]
        if t % self.B == 0:
            if not self._allocate(seq):
                return None
        else:
            last = self.blocks[seq][-1]
            if self.refcount[last] > 1:
                if len(self.free) == 0:
                    return None
                new = self.free.pop()
                self.refcount[new] = 1
                self.refcount[last] -= 1
                self.blocks[seq][-1] = new
                self.copies.append((last, new))
        blk = self.blocks[seq][t // self.B]
        self.length[seq] = t + 1
        return blk * self.B + t % self.B

    def append_tokens(self, requests):
        """requests: list of (seq, n_tokens).  Returns the slots written, in
        request order, or None (and no change) if the pool runs out."""
        saved = copy.deepcopy((self.free, self.refcount, self.blocks, self.length, self.copies))
        slots = []
        for seq, n in requests:
            for _ in range(n):
                s = self._append_one(seq)
                if s is None:
                    (self.free, self.refcount, self.blocks, self.length, self.copies) = saved
                    return None
                slots.append(s)
        return slots

    def add_sequence(self, seq, num_tokens: int):
        self.blocks[seq] = []
        self.length[seq] = 0
        slots = self.append_tokens([(seq, num_tokens)])
        if slots is None:
            del self.blocks[seq]
            del self.length[seq]
        return slots

    def take_copies(self):
        c, self.copies = self.copies, []
        return c

    def table(self, seq):
        return list(self.blocks[seq])
