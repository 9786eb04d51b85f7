"""KV-cache size arithmetic.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

Two factors of the pages' own formulas are kept apart: 2 tensors (K and V)
and the bytes per element.  The ontq page (section 2) prints the formula with
an extra factor of 2 ("2 x 2 x layers x heads x d x s x BytesPerPrecision");
its own worked numbers (about 2.6 MB per token for 80 layers x 64 heads x
128 at 16 bits) only fit 2 x layers x heads x d x bytes, which is also the
letsbuildsolutions "KV Caches" formula and thewebvale section 1 ("2 x 2 x L
x n_kv x d" with the second 2 being the two bytes).  That reading is used.
"""

from __future__ import annotations


def kv_bytes_per_token(layers: int, kv_heads: int, head_dim: int, bytes_per_elem: int) -> int:
    """K and V of one token across all layers."""
    return 2 * layers * kv_heads * head_dim * bytes_per_elem


def kv_bytes_per_layer(seq_len: int, kv_heads: int, head_dim: int, bytes_per_elem: int) -> int:
    """K and V of one layer for a whole sequence."""
    return 2 * seq_len * kv_heads * head_dim * bytes_per_elem


def kv_bytes(layers: int, kv_heads: int, head_dim: int, bytes_per_elem: int, seq_len: int) -> int:
    return kv_bytes_per_token(layers, kv_heads, head_dim, bytes_per_elem) * seq_len


def blocks_needed(num_tokens: int, block_size: int) -> int:
    """Blocks a sequence of num_tokens occupies under on-demand allocation."""
    return -(-num_tokens // block_size)


def wasted_slots(num_tokens: int, block_size: int) -> int:
    """Unused slots in a sequence's last block (internal fragmentation)."""
    return blocks_needed(num_tokens, block_size) * block_size - num_tokens
