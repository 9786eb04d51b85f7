"""Byte-exact KV-cache writes: appending new tokens and copying whole blocks.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

  * Append: a new token's key and value go to the slot the block table
    assigns it -- block ``table[t // B]``, offset ``t % B`` (thewebvale
    section 2, "The Block Table"; on-demand allocation, ontq section 3).  A
    flat slot id is ``block * B + offset``; reading taken: a negative slot
    means "skip this row" (padding).
  * Copy-on-write: when a sequence that shares a block writes a divergent
    token, the block is cloned and only that block (ontq section 3,
    "Copy-on-Write Memory Sharing"; thewebvale section 2).  Reading taken: the
    whole block (all B slots, every KV head, K and V) is copied, and every
    copy in one call reads the state from before the call.

Both functions work on the raw 16-bit patterns (int16 views), so the result
is compared bit for bit.
"""

from __future__ import annotations

import numpy as np


def bits(x) -> np.ndarray:
    """Raw 16-bit view of a torch tensor (fp16 / bf16) or array, on host."""
    if hasattr(x, "detach"):
        import torch
        return x.detach().to("cpu").contiguous().view(torch.int16).numpy().copy()
    return np.asarray(x).view(np.int16).copy()


def slot_of(block_table_row, t: int, block_size: int) -> int:
    """Flat pool slot of token position t: table[t // B] * B + t % B."""
    return int(block_table_row[t // block_size]) * block_size + t % block_size


def append_ref(k_bits, v_bits, k_new_bits, v_new_bits, slot_mapping, block_size: int):
    """Return new (k, v) pools with row i of k_new / v_new written to slot
    ``slot_mapping[i]`` for every KV head; negative slots are skipped.
    Pools [NB, Hkv, B, d] and new rows [T, Hkv, d], as int16 bit patterns."""
    k = np.array(k_bits, copy=True)
    v = np.array(v_bits, copy=True)
    for i, slot in enumerate(np.asarray(slot_mapping, dtype=np.int64)):
        if slot < 0:
            continue
        blk, off = int(slot) // block_size, int(slot) % block_size
        k[blk, :, off, :] = k_new_bits[i]
        v[blk, :, off, :] = v_new_bits[i]
    return k, v


def copy_ref(k_bits, v_bits, pairs):
    """Return new (k, v) pools where block dst holds what block src held
    before the call, for each (src, dst) pair."""
    k0 = np.array(k_bits, copy=True)
    v0 = np.array(v_bits, copy=True)
    k = np.array(k_bits, copy=True)
    v = np.array(v_bits, copy=True)
    for src, dst in np.asarray(pairs, dtype=np.int64).reshape(-1, 2):
        k[dst] = k0[src]
        v[dst] = v0[src]
    return k, v
