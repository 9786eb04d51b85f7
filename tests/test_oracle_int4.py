"""Pins for the 4-bit cache oracle: hand-worked quantisation, ties to even,
the error bound, the nibble layout byte by byte, and the append round trip."""

import numpy as np
import pytest

from oracle.int4 import (append_int4_ref, dequantize_rows, dequantized_pools, nibble_position, pack_row,
                         piece_bytes, quantize_rows, split_piece, unpack_row)


def test_hand_worked_row():
    x = np.array([7.0, -3.5, 0.4, 2.5, -7.0, 1.5, 0.0, -0.5], dtype=np.float32)
    codes, scale = quantize_rows(x)
    assert scale == np.float32(1.0)
    # 2.5 and -0.5 are ties: to the even integers 2 and -0; -3.5 -> -4; 1.5 -> 2
    np.testing.assert_array_equal(codes, [7, -4, 0, 2, -7, 2, 0, 0])
    codes, scale = quantize_rows(x * 2)
    assert scale == np.float32(2.0)
    np.testing.assert_array_equal(codes, [7, -4, 0, 2, -7, 2, 0, 0])


def test_zero_row_and_representable_values():
    codes, scale = quantize_rows(np.zeros(16, dtype=np.float32))
    assert scale == 0 and not codes.any()
    r = np.random.Generator(np.random.PCG64(1))
    c = r.integers(-7, 8, size=(5, 32)).astype(np.float32)
    c[:, 0] = 7                                            # amax code 7 in every row
    x = c * np.float32(0.375)
    codes, scale = quantize_rows(x)
    np.testing.assert_array_equal(scale, np.float32(0.375))
    np.testing.assert_array_equal(codes, c.astype(np.int8))
    np.testing.assert_array_equal(dequantize_rows(codes, scale), x.astype(np.float64))


def test_error_bound_and_range():
    r = np.random.Generator(np.random.PCG64(2))
    x = (r.standard_normal((200, 128)) * r.uniform(0.01, 100, size=(200, 1))).astype(np.float32)
    codes, scale = quantize_rows(x)
    assert codes.min() >= -7 and codes.max() <= 7            # symmetric scale: -8 never needed
    err = np.abs(dequantize_rows(codes, scale) - x)
    assert (err <= scale[:, None].astype(np.float64) * (0.5 + 1e-6)).all()
    assert (np.abs(codes).max(axis=1) == 7).all()


def test_nibble_layout_bytes():
    assert [nibble_position(e) for e in range(8)] == [0, 4, 1, 5, 2, 6, 3, 7]
    codes = np.arange(-8, 8, dtype=np.int8)                # nibbles 0..15
    b = pack_row(codes)
    # word 0 holds elements 0..7 = nibbles 0..7: even elements low, odd high
    w0 = int(np.frombuffer(b[:4].tobytes(), dtype=np.uint32)[0])
    assert w0 == (0 | 2 << 4 | 4 << 8 | 6 << 12 | 1 << 16 | 3 << 20 | 5 << 24 | 7 << 28)
    np.testing.assert_array_equal(unpack_row(b), codes)
    r = np.random.Generator(np.random.PCG64(3))
    c = r.integers(-8, 8, size=64).astype(np.int8)
    np.testing.assert_array_equal(unpack_row(pack_row(c)), c)


def test_append_round_trip_and_layout():
    r = np.random.Generator(np.random.PCG64(4))
    NB, Hkv, B, d = 4, 2, 8, 16
    P = piece_bytes(B, d)
    assert P == B * d + 8 * B
    pool = r.integers(0, 256, size=(NB, Hkv, P)).astype(np.uint8)
    kn = r.standard_normal((3, Hkv, d)).astype(np.float32)
    vn = r.standard_normal((3, Hkv, d)).astype(np.float32)
    slots = [2 * B + 5, 0 * B + 7, -1]
    p2 = append_int4_ref(pool, kn, vn, slots, B)
    kf, vf = dequantized_pools(p2, B, d)
    for i, slot in enumerate(slots[:2]):
        blk, off = slot // B, slot % B
        for h in range(Hkv):
            kq, ks = quantize_rows(kn[i, h])
            vq, vs = quantize_rows(vn[i, h])
            np.testing.assert_array_equal(kf[blk, h, off], dequantize_rows(kq, ks))
            np.testing.assert_array_equal(vf[blk, h, off], dequantize_rows(vq, vs))
    # the V half is dims-first: dim j's row of B nibbles holds token off at element off
    K, V, ks, vs = split_piece(p2[2, 1], B, d)
    vq, _ = quantize_rows(vn[0, 1])
    row0 = unpack_row(p2[2, 1][B * d // 2: B * d // 2 + B // 2])
    assert row0[5] == vq[0]
    # untouched slots keep their bytes' meaning
    K0, V0, ks0, vs0 = split_piece(pool[2, 1], B, d)
    np.testing.assert_array_equal(np.delete(V, 5, axis=0), np.delete(V0, 5, axis=0))
    np.testing.assert_array_equal(np.delete(ks, 5), np.delete(ks0, 5))
    np.testing.assert_array_equal(p2[1], pool[1])           # block 1 untouched


def test_representable_values_give_the_16_bit_attention():
    from oracle.attention import decode_ref
    r = np.random.Generator(np.random.PCG64(5))
    NB, Hkv, B, d, ctx = 3, 1, 8, 16, 19
    row = [2, 0, 1]
    kc = r.integers(-7, 8, size=(ctx, Hkv, d)).astype(np.float32)
    vc = r.integers(-7, 8, size=(ctx, Hkv, d)).astype(np.float32)
    kc[..., 0] = 7
    vc[..., 0] = -7
    kx, vx = kc * np.float32(0.25), vc * np.float32(0.5)
    pool = np.zeros((NB, Hkv, piece_bytes(B, d)), np.uint8)
    slots = [row[t // B] * B + t % B for t in range(ctx)]
    pool = append_int4_ref(pool, kx, vx, slots, B)
    kf, vf = dequantized_pools(pool, B, d)
    kd = np.zeros((NB, Hkv, B, d))
    vd = np.zeros((NB, Hkv, B, d))
    for t in range(ctx):
        kd[row[t // B], :, t % B] = kx[t]
        vd[row[t // B], :, t % B] = vx[t]
    q = r.standard_normal((1, 2, d))
    a = decode_ref(q, kf, vf, np.array([row]), np.array([ctx]), 0.3)
    b = decode_ref(q, kd, vd, np.array([row]), np.array([ctx]), 0.3)
    np.testing.assert_array_equal(a, b)
