"""4-bit integer KV cache: symmetric codes with one scale per cached row.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

The pages: compressing the KV cache to 4 bits (INT4) quadruples how many
requests fit (ontq "AI Inference Serving at Scale", section 6); 4-bit integer
formats carry per-group scaling factors (letsbuildsolutions "How LLM Inference
Engines Work", quantization section, on 4-bit weight formats).  They give no
bit layout.  Readings taken:

  * A group is one cached row: the d values of one (token, KV head) of K, or
    of V.  Its scale is s = amax / 7 (amax = the largest magnitude, one fp32
    division); the codes are the nearest integers to x / s (one fp32 division
    each, ties to even), clamped to [-8, 7].  A row of zeros has s = 0 and
    codes 0.  Decoding: x' = code * s.
  * Layout of the pool: bytes [blocks][kv heads][piece]; each (block, head)
    piece holds, in order, the K codes token-major ([B][d] nibbles), the V
    codes dims-first ([d][B] nibbles), the B fp32 K scales and the B fp32 V
    scales.  Codes are stored as nibbles code + 8, packed along the row in
    32-bit little-endian words of 8 elements: element 2k of a word in nibble
    k, element 2k + 1 in nibble k + 4.

Everything below follows those definitions literally.
"""

from __future__ import annotations

import numpy as np


def quantize_rows(x):
    """x [..., d] (fp32 values) -> (codes int8 [..., d], scales fp32 [...])."""
    xf = np.asarray(x, dtype=np.float32)
    amax = np.abs(xf).max(axis=-1)
    scale = (amax / np.float32(7.0)).astype(np.float32)
    safe = np.where(scale > 0, scale, np.float32(1.0)).astype(np.float32)
    q = np.rint(xf / safe[..., None])                  # fp32 division; rint: ties to even
    q = np.where(scale[..., None] > 0, q, 0.0)
    return np.clip(q, -8, 7).astype(np.int8), scale


def dequantize_rows(codes, scales):
    """fp64 values code * scale (garbage scale bytes give inf / NaN rows)."""
    with np.errstate(invalid="ignore", over="ignore"):
        return np.asarray(codes, dtype=np.float64) * np.asarray(scales, dtype=np.float64)[..., None]


def nibble_position(e: int) -> int:
    """Nibble (0..7) of element e (0..7) inside its 32-bit word."""
    return e // 2 if e % 2 == 0 else 4 + e // 2


def pack_row(codes) -> np.ndarray:
    """int8 codes [n] (n a multiple of 8) -> n / 2 bytes (little-endian words)."""
    c = np.asarray(codes, dtype=np.int64)
    n = c.size
    assert n % 8 == 0
    out = np.zeros(n // 2, dtype=np.uint8)
    for w in range(n // 8):
        word = 0
        for e in range(8):
            word |= (int(c[8 * w + e]) + 8) << (4 * nibble_position(e))
        out[4 * w:4 * w + 4] = np.frombuffer(np.uint32(word).tobytes(), dtype=np.uint8)
    return out


def unpack_row(b) -> np.ndarray:
    """n / 2 bytes -> int8 codes [n] (inverse of pack_row)."""
    b = np.asarray(b, dtype=np.uint8)
    n = 2 * b.size
    out = np.zeros(n, dtype=np.int8)
    for w in range(n // 8):
        word = int(np.frombuffer(b[4 * w:4 * w + 4].tobytes(), dtype=np.uint32)[0])
        for e in range(8):
            out[8 * w + e] = ((word >> (4 * nibble_position(e))) & 0xF) - 8
    return out


def piece_bytes(block_size: int, d: int) -> int:
    return block_size * d // 2 * 2 + 2 * block_size * 4


def _offsets(B, d):
    kc = 0
    vc = B * d // 2
    ks = vc + d * B // 2
    vs = ks + 4 * B
    return kc, vc, ks, vs


def split_piece(piece, B, d):
    """One piece's bytes -> (K codes [B][d], V codes [B][d] token-major,
    K scales [B], V scales [B])."""
    p = np.asarray(piece, dtype=np.uint8)
    kc, vc, ks, vs = _offsets(B, d)
    K = np.stack([unpack_row(p[kc + t * d // 2: kc + (t + 1) * d // 2]) for t in range(B)])
    Vt = np.stack([unpack_row(p[vc + j * B // 2: vc + (j + 1) * B // 2]) for j in range(d)])   # [d][B]
    kscale = np.frombuffer(p[ks:ks + 4 * B].tobytes(), dtype=np.float32).copy()
    vscale = np.frombuffer(p[vs:vs + 4 * B].tobytes(), dtype=np.float32).copy()
    return K, Vt.T.copy(), kscale, vscale


def dequantized_pools(pool, B, d):
    """Pool bytes [NB][Hkv][piece] -> fp64 K, V pools [NB][Hkv][B][d]."""
    p = np.asarray(pool, dtype=np.uint8)
    NB, Hkv = p.shape[0], p.shape[1]
    kf = np.zeros((NB, Hkv, B, d))
    vf = np.zeros((NB, Hkv, B, d))
    for b in range(NB):
        for h in range(Hkv):
            K, V, ks, vs = split_piece(p[b, h], B, d)
            kf[b, h] = dequantize_rows(K, ks)
            vf[b, h] = dequantize_rows(V, vs)
    return kf, vf


def append_int4_ref(pool, k_new, v_new, slot_mapping, B):
    """New pool bytes with row i of k_new / v_new (fp32 values [T, Hkv, d])
    quantized into slot slot_mapping[i]; negative slots skip."""
    p = np.array(pool, dtype=np.uint8, copy=True)
    kn = np.asarray(k_new, dtype=np.float32)
    vn = np.asarray(v_new, dtype=np.float32)
    T, Hkv, d = kn.shape
    kc, vc, ks, vs = _offsets(B, d)
    for i, slot in enumerate(np.asarray(slot_mapping, dtype=np.int64)):
        if slot < 0:
            continue
        blk, off = int(slot) // B, int(slot) % B
        kq, ksc = quantize_rows(kn[i])
        vq, vsc = quantize_rows(vn[i])
        for h in range(Hkv):
            piece = p[blk, h]
            piece[kc + off * d // 2: kc + (off + 1) * d // 2] = pack_row(kq[h])
            for j in range(d):
                row = piece[vc + j * B // 2: vc + (j + 1) * B // 2]
                codes = unpack_row(row)
                codes[off] = vq[h, j]
                piece[vc + j * B // 2: vc + (j + 1) * B // 2] = pack_row(codes)
            piece[ks + 4 * off: ks + 4 * off + 4] = np.frombuffer(np.float32(ksc[h]).tobytes(), dtype=np.uint8)
            piece[vs + 4 * off: vs + 4 * off + 4] = np.frombuffer(np.float32(vsc[h]).tobytes(), dtype=np.uint8)
    return p
