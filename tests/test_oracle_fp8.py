"""Pins for the FP8 encodings of the oracle: every code, the formats' known
constants, rounding ties, saturation."""

import numpy as np
import pytest

from oracle.fp8 import decode_code, encode_value, max_finite, quantize, dequantize


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_every_finite_code_round_trips(fmt):
    for c in range(256):
        v = decode_code(c, fmt)
        if np.isfinite(v):
            got = encode_value(v, fmt)
            assert decode_code(got, fmt) == v and (got == c or v == 0.0), (c, v, got)


def test_known_constants():
    assert max_finite("e4m3") == 448.0
    assert max_finite("e5m2") == 57344.0
    assert decode_code(0x01, "e4m3") == 2.0 ** -9          # smallest subnormal
    assert decode_code(0x08, "e4m3") == 2.0 ** -6          # smallest normal
    assert decode_code(0x7E, "e4m3") == 448.0
    assert np.isnan(decode_code(0x7F, "e4m3")) and np.isnan(decode_code(0xFF, "e4m3"))
    assert decode_code(0x38, "e4m3") == 1.0
    assert decode_code(0x3C, "e5m2") == 1.0
    assert decode_code(0x7C, "e5m2") == np.inf
    assert decode_code(0x01, "e5m2") == 2.0 ** -16
    assert decode_code(0xC0, "e4m3") == -2.0


def test_ties_go_to_even_and_saturation():
    # 1.0 = 0x38 and 1.125 = 0x39 in E4M3: the midpoint 1.0625 goes to 0x38 (even)
    assert encode_value(1.0625, "e4m3") == 0x38
    # 1.125 (0x39) and 1.25 (0x3A): midpoint 1.1875 goes to 0x3A
    assert encode_value(1.1875, "e4m3") == 0x3A
    assert encode_value(1.19, "e4m3") == 0x3A and encode_value(1.18, "e4m3") == 0x39
    assert encode_value(1e6, "e4m3") == 0x7E and encode_value(-1e6, "e4m3") == 0xFE
    assert encode_value(1e9, "e5m2") == 0x7B                # largest finite, not inf
    assert encode_value(2.0 ** -12, "e4m3") == 0x00         # below half the smallest subnormal
    assert encode_value(3 * 2.0 ** -10, "e4m3") == 0x02     # 1.5 subnormal steps: tie -> even code
    assert encode_value(5 * 2.0 ** -10, "e4m3") == 0x02     # 2.5 steps: tie -> even code
    assert np.isnan(decode_code(encode_value(float("nan"), "e4m3"), "e4m3"))


def test_quantize_divides_by_the_scale_in_fp32():
    x = np.array([0.5, -3.0, 100.0, 7.0e-4], dtype=np.float32)
    codes = quantize(x, 0.25, "e4m3")
    # 100 / 0.25 = 400 lies halfway between 384 and 416: the even code (384)
    np.testing.assert_array_equal(dequantize(codes, 0.25, "e4m3"), [0.5, -3.0, 96.0, 0.25 * 2.0 ** -9])


def test_append_then_dequantize_returns_the_quantized_rows():
    from oracle.fp8 import append_fp8_ref, dequantized_pools, split_pool
    from oracle.attention import gather_sequence
    r = np.random.Generator(np.random.PCG64(1))
    NB, Hkv, B, d = 6, 2, 4, 8
    kv = r.integers(0, 0x7E, size=(NB, Hkv, 2, B * d)).astype(np.uint8)
    kn = r.standard_normal((3, Hkv, d)).astype(np.float32)
    vn = r.standard_normal((3, Hkv, d)).astype(np.float32)
    row = [4, 1]
    slots = [4 * 4 + 0, 1 * 4 + 3, -1]
    kv2 = append_fp8_ref(kv, kn, vn, slots, B, 0.5, 2.0, "e4m3")
    kf, vf = dequantized_pools(kv2, B, 0.5, 2.0, "e4m3")
    K, V = gather_sequence(kf, vf, row, 8, 1, B)
    np.testing.assert_array_equal(K[0], dequantize(quantize(kn[0, 1], 0.5, "e4m3"), 0.5, "e4m3"))
    np.testing.assert_array_equal(V[7], dequantize(quantize(vn[1, 1], 2.0, "e4m3"), 2.0, "e4m3"))
    # untouched slots keep their codes; the V half of a piece is dims-first
    k0, v0 = split_pool(kv, B)
    k2, v2 = split_pool(kv2, B)
    np.testing.assert_array_equal(v2[4, :, :, 1:], v0[4, :, :, 1:])
    np.testing.assert_array_equal(v2[4, 0, :, 0], quantize(vn[0, 0], 2.0, "e4m3"))
    np.testing.assert_array_equal(kv2[4, 0, 1, 0:B], [v2[4, 0, 0, t] for t in range(B)])


def test_representable_values_survive_the_8_bit_cache():
    """Values already on the E4M3 grid (times the scales) decode exactly: the
    8-bit cache then gives the 16-bit cache's attention."""
    from oracle.fp8 import append_fp8_ref, dequantized_pools
    from oracle.attention import decode_ref
    r = np.random.Generator(np.random.PCG64(2))
    NB, Hkv, B, d, ctx = 5, 1, 4, 8, 13
    grid = np.array([decode_code(c, "e4m3") for c in range(0x70)])
    kc = r.choice(grid, size=(NB, Hkv, B, d)) * 0.25
    vc = r.choice(grid, size=(NB, Hkv, B, d)) * 4.0
    row = [3, 0, 4, 1]
    slots = [row[t // B] * B + t % B for t in range(ctx)]
    kv = np.zeros((NB, Hkv, 2, B * d), np.uint8)
    kn = np.stack([kc[row[t // B], :, t % B] for t in range(ctx)])
    vn = np.stack([vc[row[t // B], :, t % B] for t in range(ctx)])
    kv = append_fp8_ref(kv, kn, vn, slots, B, 0.25, 4.0, "e4m3")
    kf, vf = dequantized_pools(kv, B, 0.25, 4.0, "e4m3")
    q = r.standard_normal((1, 2, d))
    a = decode_ref(q, kf, vf, np.array([row]), np.array([ctx]), 0.3)
    b = decode_ref(q, kc, vc, np.array([row]), np.array([ctx]), 0.3)
    np.testing.assert_array_equal(a, b)


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_array_quantizer_equals_the_scalar_rule(fmt):
    r = np.random.Generator(np.random.PCG64(3))
    x = np.concatenate([r.standard_normal(3000) * 10 ** r.uniform(-4, 3, 3000),
                        [0.0, -0.0, 1.0625, 1.1875, 3 * 2.0 ** -10, 1e6, -1e6, 447.9, 448.0, 464.0, 480.0]])
    x = x.astype(np.float32)
    want = np.array([encode_value(float(v), fmt) for v in x], dtype=np.uint8)
    np.testing.assert_array_equal(quantize(x, 1.0, fmt), want)


def test_k_rows_of_128_bytes_store_permuted_pieces():
    """d = 128: each K token row keeps its own 128 bytes, with 16-byte piece c
    of row r at piece position c XOR (r mod 8); V stays dims-first.  The
    round trip through the pool gives back exactly the quantized rows."""
    from oracle.fp8 import append_fp8_ref, dequantized_pools, k_positions, split_pool
    r = np.random.Generator(np.random.PCG64(7))
    NB, Hkv, B, d = 3, 2, 16, 128
    kv = np.zeros((NB, Hkv, 2, B * d), np.uint8)
    kn = r.standard_normal((B, Hkv, d)).astype(np.float32)
    vn = r.standard_normal((B, Hkv, d)).astype(np.float32)
    slots = [2 * B + t for t in range(B)]
    kv = append_fp8_ref(kv, kn, vn, slots, B, 0.5, 0.5, "e4m3")
    raw = kv[2, 1, 0]
    for t in (0, 1, 7, 8, 13):
        want = quantize(kn[t, 1], 0.5, "e4m3")
        row = raw[t * 128:(t + 1) * 128]
        assert sorted(row.tolist()) == sorted(want.tolist())          # the row's own bytes
        for c in range(8):
            np.testing.assert_array_equal(row[16 * (c ^ (t % 8)):16 * (c ^ (t % 8)) + 16], want[16 * c:16 * c + 16])
    assert sorted(k_positions(B, d).ravel().tolist()) == list(range(B * d))  # a permutation
    np.testing.assert_array_equal(k_positions(B, 64), np.arange(B * 64).reshape(B, 64))
    k, v = split_pool(kv, B)
    kf, vf = dequantized_pools(kv, B, 0.5, 0.5, "e4m3")
    for t in range(B):
        np.testing.assert_array_equal(k[2, 1, t], quantize(kn[t, 1], 0.5, "e4m3"))
        np.testing.assert_array_equal(v[2, 0, :, t], quantize(vn[t, 0], 0.5, "e4m3"))
        np.testing.assert_array_equal(kf[2, 0, t], dequantize(quantize(kn[t, 0], 0.5, "e4m3"), 0.5, "e4m3"))
