"""8-bit floating-point KV cache: the E4M3 and E5M2 encodings.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

The pages: storing keys and values in 8 bits (FP8) instead of 16 halves the
KV memory (ontq "AI Inference Serving at Scale", section 6); the vLLM
deployment script on thewebvale (section 5) names fp8_e5m2 as a KV-cache
dtype.  They give neither the bit layout nor a scaling rule.  Readings taken:

  * E4M3 is the OCP 8-bit format with 1 sign, 4 exponent (bias 7), 3 mantissa
    bits, subnormals, no infinities, one NaN pattern per sign (S.1111.111);
    its largest finite magnitude is 448.  E5M2 has 5 exponent bits (bias 15),
    2 mantissa bits, subnormals, infinities and NaNs, largest finite 57344.
  * A cache tensor stores code(x / s) for a per-tensor fp32 scale s (one for
    K, one for V); decoding multiplies by s.  The division is one fp32
    division, rounded to nearest.
  * Encoding rounds to the nearest representable value, ties to the even
    code, and saturates finite values beyond the largest magnitude to it;
    NaN stays NaN.

Everything below is written from those definitions: values are enumerated
from the bit fields, and encoding picks the nearest enumerated value.
"""

from __future__ import annotations

import numpy as np

FORMATS = {"e4m3": (4, 3, 7), "e5m2": (5, 2, 15)}


def decode_code(code: int, fmt: str) -> float:
    """Value of one 8-bit code (Python float; inf/nan where the format has them)."""
    e_bits, m_bits, bias = FORMATS[fmt]
    sign = -1.0 if code & 0x80 else 1.0
    e = (code >> m_bits) & ((1 << e_bits) - 1)
    m = code & ((1 << m_bits) - 1)
    e_max = (1 << e_bits) - 1
    if fmt == "e4m3":
        if e == e_max and m == (1 << m_bits) - 1:
            return float("nan")
    elif e == e_max:
        return sign * float("inf") if m == 0 else float("nan")
    if e == 0:
        return sign * (m / (1 << m_bits)) * 2.0 ** (1 - bias)
    return sign * (1.0 + m / (1 << m_bits)) * 2.0 ** (e - bias)


def _finite_table(fmt):
    """Non-negative finite codes and their values, ascending."""
    codes = [c for c in range(0x80) if np.isfinite(decode_code(c, fmt))]
    vals = [decode_code(c, fmt) for c in codes]
    order = np.argsort(vals, kind="stable")
    return np.array(codes)[order], np.array(vals)[order]


def max_finite(fmt: str) -> float:
    return float(_finite_table(fmt)[1][-1])


def encode_value(x: float, fmt: str) -> int:
    """Nearest code to x (ties to the even code), saturating to the largest
    finite magnitude; NaN -> the format's NaN code (positive sign)."""
    if np.isnan(x):
        return 0x7F
    codes, vals = _finite_table(fmt)
    a = abs(float(x))
    sign = 0x80 if (np.signbit(x) and a != 0.0) else 0
    if np.signbit(x) and a == 0.0:
        sign = 0x80
    if a >= vals[-1]:
        return sign | int(codes[-1])
    i = int(np.searchsorted(vals, a))           # vals[i-1] < a <= vals[i]
    if vals[i] == a:
        return sign | int(codes[i])
    lo, hi = i - 1, i
    dlo, dhi = a - vals[lo], vals[hi] - a
    if dlo < dhi:
        pick = lo
    elif dhi < dlo:
        pick = hi
    else:
        pick = lo if (codes[lo] & 1) == 0 else hi   # even mantissa
    return sign | int(codes[pick])


def decode_array(codes, fmt: str) -> np.ndarray:
    table = np.array([decode_code(c, fmt) for c in range(256)])
    return table[np.asarray(codes, dtype=np.uint8)]


def quantize(x, scale: float, fmt: str) -> np.ndarray:
    """Codes of x / scale (one fp32 division each) for an array of 16-bit
    values: the same nearest / ties-to-even / saturating rule as
    encode_value, applied with a sorted table of the format's values."""
    xf = np.asarray(x, dtype=np.float32) / np.float32(scale)
    codes, vals = _finite_table(fmt)
    a = np.abs(xf).astype(np.float64)
    i = np.clip(np.searchsorted(vals, a), 1, len(vals) - 1)     # vals[i-1] < a <= vals[i]
    lo, hi = i - 1, i
    dlo, dhi = a - vals[lo], vals[hi] - a
    even_lo = (codes[lo] & 1) == 0
    pick = np.where(dlo < dhi, lo, np.where(dhi < dlo, hi, np.where(even_lo, lo, hi)))
    pick = np.where(a >= vals[-1], len(vals) - 1, pick)
    out = codes[pick].astype(np.uint8) | np.where(np.signbit(xf), 0x80, 0).astype(np.uint8)
    return np.where(np.isnan(xf), np.uint8(0x7F), out).astype(np.uint8)


def dequantize(codes, scale: float, fmt: str) -> np.ndarray:
    """fp64 values of stored codes: decode(code) * scale."""
    return decode_array(codes, fmt) * float(np.float32(scale))


# ---------------------------------------------------------------------------
# The 8-bit cache.  Reading taken for the layout (the pages fix none): one
# pool of bytes [blocks][kv heads][2][B * d]; for each (block, head) the first
# half holds K codes token-major ([B][d], as the 16-bit cache) and the second
# half V codes dims-first ([d][B]), so the whole piece is contiguous.  Inside
# the K half, each 128-byte span of a token row keeps its bytes but stores its
# eight 16-byte pieces in a permuted order: piece c of row r sits at piece
# position c XOR (r mod 8).  Rows whose width is not a multiple of 128 bytes
# keep the plain order.
# ---------------------------------------------------------------------------

def k_positions(block_size: int, d: int) -> np.ndarray:
    """[B][d] index, inside a K half, of the code of (token row r, dim c)."""
    r = np.arange(block_size)[:, None]
    c = np.arange(d)[None, :]
    if d % 128:
        return r * d + c
    return r * d + (c // 128) * 128 + 16 * (((c % 128) // 16) ^ (r % 8)) + c % 16


def _flat(kv_codes):
    kv = np.asarray(kv_codes)
    if kv.ndim == 5:                         # [NB][Hkv][2][B][d] byte view of the same pool
        kv = kv.reshape(kv.shape[0], kv.shape[1], 2, -1)
    return kv


def split_pool(kv_codes, block_size):
    """(K codes [NB][Hkv][B][d], V codes [NB][Hkv][d][B]) of a pool; K is a
    gathered copy (the row pieces put back in order), V a view."""
    kv = _flat(kv_codes)
    NB, Hkv, two, n = kv.shape
    d = n // block_size
    k = kv[:, :, 0][..., k_positions(block_size, d)]
    return k, kv[:, :, 1].reshape(NB, Hkv, d, block_size)


def append_fp8_ref(kv_codes, k_new, v_new, slot_mapping, block_size, k_scale, v_scale, fmt):
    """New pool with row i of k_new / v_new (16-bit values [T, Hkv, d])
    quantized into slot slot_mapping[i]; negative slots skip."""
    kv = np.array(_flat(kv_codes), copy=True)
    NB, Hkv, two, n = kv.shape
    d = n // block_size
    pos = k_positions(block_size, d)
    v = kv[:, :, 1].reshape(NB, Hkv, d, block_size)
    kn = np.asarray(k_new, dtype=np.float32)
    vn = np.asarray(v_new, dtype=np.float32)
    for i, slot in enumerate(np.asarray(slot_mapping, dtype=np.int64)):
        if slot < 0:
            continue
        blk, off = int(slot) // block_size, int(slot) % block_size
        khalf = kv[blk, :, 0]                # [Hkv][B * d] view
        khalf[:, pos[off]] = quantize(kn[i], k_scale, fmt)
        v[blk, :, :, off] = quantize(vn[i], v_scale, fmt)
    return kv


def dequantized_pools(kv_codes, block_size, k_scale, v_scale, fmt):
    """fp64 K and V pools in the 16-bit cache's layout [blocks][kv heads][B][d]."""
    k, v = split_pool(kv_codes, block_size)
    return dequantize(k, k_scale, fmt), dequantize(np.swapaxes(v, 2, 3), v_scale, fmt)
