"""Host-side block manager: free list, per-block refcounts, on-demand
allocation, fork and copy-on-write.  It builds the block tables, context
lengths, slot mappings and copy lists that the kernels consume; it does no
math on keys or values.

Semantics (the pages' BlockManager and its surroundings):
  * The free list is a stack: allocation pops its end and gives the block
    refcount 1; freeing a sequence decrements each of its blocks and pushes a
    block back when its count reaches 0; allocation on an empty list fails
    ("How LLM Inference Engines Work ...", letsbuildsolutions, section
    "PagedAttention: Virtual Memory for KV Caches").
  * A block is taken only when the previous one is full -- just before token
    t with t % B == 0 is written (ontq "AI Inference Serving at Scale",
    section 3, on-demand allocation).
  * fork() makes a child point at its parent's blocks.  Writing into a block
    whose refcount is above 1 takes a fresh block, queues a whole-block copy
    (old -> new) and drops one reference to the old block; a writer that finds
    refcount 1 writes in place (ontq section 3 copy-on-write; thewebvale
    section 2).  Requests in one call are served in the order given.
  * A multi-token request succeeds as a whole or changes nothing, and reports
    failure by returning None.
  * Slot of token t: table[t // B] * B + t % B (thewebvale section 2).
"""

from __future__ import annotations

from typing import Dict, Iterable, List, Optional, Sequence, Tuple

import numpy as np


class BlockManager:
    def __init__(self, num_blocks: int, block_size: int, free_order: Optional[Sequence[int]] = None,
                 seed: Optional[int] = None):
        if num_blocks <= 0 or block_size <= 0:
            raise ValueError("num_blocks and block_size must be positive")
        self.num_blocks = int(num_blocks)
        self.block_size = int(block_size)
        if free_order is None:
            if seed is None:
                free_order = np.arange(num_blocks)
            else:
                free_order = np.random.Generator(np.random.PCG64(seed)).permutation(num_blocks)
        free_order = [int(b) for b in free_order]
        if sorted(free_order) != list(range(num_blocks)):
            raise ValueError("free_order must be a permutation of range(num_blocks)")
        self._free: List[int] = free_order
        self._ref = np.zeros(num_blocks, dtype=np.int32)
        self._blocks: Dict[object, List[int]] = {}
        self._len: Dict[object, int] = {}
        self._copies: List[Tuple[int, int]] = []

    # ------------------------------------------------------------ queries
    @property
    def num_free(self) -> int:
        return len(self._free)

    @property
    def num_used(self) -> int:
        return self.num_blocks - len(self._free)

    def sequences(self) -> List[object]:
        return list(self._blocks)

    def length(self, seq) -> int:
        return self._len[seq]

    def table(self, seq) -> List[int]:
        return list(self._blocks[seq])

    def refcount(self, block: int) -> int:
        return int(self._ref[block])

    def free_blocks(self) -> List[int]:
        return list(self._free)

    def block_tables(self, seqs: Sequence, max_blocks: int, pad: int = -1) -> np.ndarray:
        out = np.full((len(seqs), max_blocks), pad, dtype=np.int32)
        for i, s in enumerate(seqs):
            b = self._blocks[s]
            if len(b) > max_blocks:
                raise ValueError(f"sequence {s!r} has {len(b)} blocks > max_blocks {max_blocks}")
            out[i, :len(b)] = b
        return out

    def shared_prefix_groups(self, seqs: Sequence, min_members: int = 2):
        """Find runs of consecutive sequences (in batch order) whose tables
        begin with the same full blocks, for prefix-aware decode.

        Returns (group_starts [G + 1], group_prefix_blocks [G]) as int32
        arrays: group i is seqs[group_starts[i]:group_starts[i + 1]] and its
        members share their first group_prefix_blocks[i] blocks, each
        completely filled in every member.  Gaps between runs become groups
        with no shared blocks, so the boundaries stay contiguous."""
        B = self.block_size
        runs = []
        i, n = 0, len(seqs)
        while i < n:
            first = self._blocks[seqs[i]]
            j = i + 1
            while j < n and first and self._blocks[seqs[j]][:1] == first[:1]:
                j += 1
            if j - i >= min_members:
                p = min(self._len[s] for s in seqs[i:j]) // B
                for s in seqs[i + 1:j]:
                    b = self._blocks[s]
                    k = 0
                    while k < p and b[k] == first[k]:
                        k += 1
                    p = k
                if p > 0:
                    runs.append((i, j, p))
            i = j
        bounds, prefix = [], []
        for a, b, p in runs:
            if bounds and bounds[-1] < a:
                prefix.append(0)
                bounds.append(a)
            elif not bounds:
                bounds.append(a)
            prefix.append(p)
            bounds.append(b)
        if not bounds:
            bounds = [0]
        return np.asarray(bounds, dtype=np.int32), np.asarray(prefix, dtype=np.int32)

    def context_lens(self, seqs: Sequence) -> np.ndarray:
        return np.array([self._len[s] for s in seqs], dtype=np.int32)

    def stats(self) -> dict:
        """Pool utilisation, internal fragmentation and sharing."""
        logical = sum(len(b) for b in self._blocks.values())
        tokens = sum(self._len.values())
        used = self.num_used
        slots = used * self.block_size
        unique_tokens = 0
        seen = set()
        for s, blocks in self._blocks.items():
            n = self._len[s]
            for i, b in enumerate(blocks):
                if b in seen:
                    continue
                seen.add(b)
                unique_tokens += min(self.block_size, n - i * self.block_size)
        return {
            "blocks_used": used,
            "blocks_free": len(self._free),
            "utilization": used / self.num_blocks,
            "logical_blocks": logical,
            "sharing_ratio": (logical / used) if used else 1.0,
            "tokens": tokens,
            "internal_waste_slots": slots - unique_tokens,
            "fragmentation": ((slots - unique_tokens) / slots) if slots else 0.0,
        }

    # ------------------------------------------------------------ mutation
    def _pop(self) -> int:
        b = self._free.pop()
        self._ref[b] = 1
        return b

    def _blocks_needed(self, requests: Iterable[Tuple[object, int]]) -> int:
        """Free blocks the requests will take, replaying copy-on-write
        decisions on a scratch view of lengths and refcounts."""
        B = self.block_size
        lens: Dict[object, int] = {}
        private: Dict[object, bool] = {}
        ref_delta: Dict[int, int] = {}
        need = 0
        for seq, n in requests:
            if n <= 0:
                continue
            t = lens.get(seq, self._len[seq])
            if t % B != 0 and not private.get(seq, False):
                last = self._blocks[seq][-1]
                if self._ref[last] + ref_delta.get(last, 0) > 1:
                    need += 1
                    ref_delta[last] = ref_delta.get(last, 0) - 1
            private[seq] = True
            need += -(-(t + n) // B) - (-(-t // B))
            lens[seq] = t + n
        return need

    def append_slots(self, requests) -> Optional[np.ndarray]:
        """Reserve slots for new tokens.

        ``requests`` is a list of (seq, n_tokens), or a list of sequence ids
        (one token each).  Returns the int64 slots in request order, or None
        (nothing changed) if the pool cannot hold them.  Copy-on-write copies
        are queued; fetch them with ``take_copies()``.
        """
        reqs = [(r, 1) if not isinstance(r, tuple) else (r[0], int(r[1])) for r in requests]
        for seq, n in reqs:
            if seq not in self._blocks:
                raise KeyError(f"unknown sequence {seq!r}")
            if n < 0:
                raise ValueError("negative token count")
        if self._blocks_needed(reqs) > len(self._free):
            return None
        B = self.block_size
        out = np.empty(sum(n for _, n in reqs), dtype=np.int64)
        pos = 0
        for seq, n in reqs:
            if n == 0:
                continue
            blocks = self._blocks[seq]
            t = self._len[seq]
            if t % B != 0:
                last = blocks[-1]
                if self._ref[last] > 1:
                    new = self._pop()
                    self._ref[last] -= 1
                    blocks[-1] = new
                    self._copies.append((last, new))
            for _ in range(-(-(t + n) // B) - len(blocks)):
                blocks.append(self._pop())
            # only the blocks the new tokens land in: O(n), not O(context)
            if n == 1:
                out[pos] = blocks[t // B] * B + t % B
            else:
                b0 = t // B
                tt = np.arange(t, t + n, dtype=np.int64)
                tbl = np.asarray(blocks[b0:(t + n - 1) // B + 1], dtype=np.int64)
                out[pos:pos + n] = tbl[tt // B - b0] * B + tt % B
            pos += n
            self._len[seq] = t + n
        return out

    def add_sequence(self, seq, num_tokens: int) -> Optional[np.ndarray]:
        """Start a sequence and reserve slots for its first num_tokens tokens."""
        if seq in self._blocks:
            raise KeyError(f"sequence {seq!r} exists")
        self._blocks[seq] = []
        self._len[seq] = 0
        slots = self.append_slots([(seq, int(num_tokens))])
        if slots is None:
            del self._blocks[seq]
            del self._len[seq]
        return slots

    def fork(self, parent, child) -> None:
        """Child shares every block of parent (refcount + 1 each)."""
        if child in self._blocks:
            raise KeyError(f"sequence {child!r} exists")
        blocks = self._blocks[parent]
        self._blocks[child] = list(blocks)
        self._len[child] = self._len[parent]
        if blocks:
            np.add.at(self._ref, np.asarray(blocks), 1)

    def free(self, seq) -> None:
        """Drop a finished sequence; blocks reaching refcount 0 go back to the free list."""
        for b in self._blocks.pop(seq):
            self._ref[b] -= 1
            if self._ref[b] == 0:
                self._free.append(b)
        del self._len[seq]

    def take_copies(self) -> np.ndarray:
        """Queued (src, dst) copy-on-write pairs as int32 [n, 2]; clears the queue."""
        c = np.asarray(self._copies, dtype=np.int32).reshape(-1, 2)
        self._copies = []
        return c

    # ------------------------------------------------------------ state
    def snapshot(self) -> dict:
        return {
            "num_blocks": self.num_blocks, "block_size": self.block_size, "free": list(self._free),
            "ref": self._ref.tolist(), "blocks": {k: list(v) for k, v in self._blocks.items()},
            "len": dict(self._len), "copies": list(self._copies),
        }

    @classmethod
    def restore(cls, snap: dict) -> "BlockManager":
        bm = cls(snap["num_blocks"], snap["block_size"])
        bm._free = list(snap["free"])
        bm._ref = np.asarray(snap["ref"], dtype=np.int32)
        bm._blocks = {k: list(v) for k, v in snap["blocks"].items()}
        bm._len = dict(snap["len"])
        bm._copies = [tuple(c) for c in snap["copies"]]
        return bm
