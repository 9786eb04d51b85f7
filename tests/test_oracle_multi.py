"""Pins for the multi-token query oracle: it reduces to decode for one token,
to the last rows of textbook causal attention over the un-paged sequence, to
v_0 for the first token of a sequence, to pure-Python brute force, and to
MHA with repeated KV heads."""

import numpy as np
import pytest

from oracle.attention import causal_dense_ref, decode_multi_ref, decode_ref


def paged_case(r, N, Hq, Hkv, d, B, ctx, NB=None, dtype=np.float64):
    MB = max(1, max(-(-c // B) for c in ctx))
    NB = NB or N * MB + 3
    k = r.standard_normal((NB, Hkv, B, d))
    v = r.standard_normal((NB, Hkv, B, d))
    ids = r.permutation(NB)
    tables = np.full((N, MB), -1, np.int64)
    pos = 0
    for b, c in enumerate(ctx):
        nb = -(-c // B)
        tables[b, :nb] = ids[pos:pos + nb]
        pos += nb
    return k, v, tables


def test_one_token_chunks_equal_decode():
    r = np.random.Generator(np.random.PCG64(11))
    N, Hq, Hkv, d, B = 5, 8, 2, 16, 4
    ctx = [1, 7, 12, 4, 9]
    k, v, tables = paged_case(r, N, Hq, Hkv, d, B, ctx)
    q = r.standard_normal((N, Hq, d))
    qs = np.arange(N + 1)
    a = decode_multi_ref(q, k, v, tables, ctx, qs, 0.37)
    b = decode_ref(q, k, v, tables, ctx, 0.37)
    np.testing.assert_allclose(a, b, rtol=0, atol=1e-13)


@pytest.mark.parametrize("n", [1, 3, 8])
def test_equals_last_rows_of_causal_attention(n):
    r = np.random.Generator(np.random.PCG64(20 + n))
    Hq, Hkv, d, B, ctx = 6, 3, 8, 4, 11
    k_seq = r.standard_normal((ctx, Hkv, d))
    v_seq = r.standard_normal((ctx, Hkv, d))
    q_all = r.standard_normal((ctx, Hq, d))
    dense = causal_dense_ref(q_all, k_seq, v_seq, 0.5)
    # the same sequence, paged: token t at block ids[t // B], offset t % B
    nb = -(-ctx // B)
    NB = nb + 4
    ids = r.permutation(NB)[:nb]
    kp = np.full((NB, Hkv, B, d), np.nan)
    vp = np.full((NB, Hkv, B, d), np.nan)
    for t in range(ctx):
        kp[ids[t // B], :, t % B] = k_seq[t]
        vp[ids[t // B], :, t % B] = v_seq[t]
    got = decode_multi_ref(q_all[ctx - n:], kp, vp, ids[None, :], [ctx], [0, n], 0.5)
    np.testing.assert_allclose(got, dense[ctx - n:], rtol=0, atol=1e-12)


def test_first_token_of_a_sequence_sees_only_itself():
    # a prefill chunk from the start: ctx == q_len, token 0 attends to key 0 alone
    r = np.random.Generator(np.random.PCG64(31))
    Hq, Hkv, d, B, n = 4, 4, 8, 4, 6
    k, v, tables = paged_case(r, 1, Hq, Hkv, d, B, [n])
    q = r.standard_normal((n, Hq, d)) * 10
    out = decode_multi_ref(q, k, v, tables, [n], [0, n], 1.0)
    blk = tables[0, 0]
    for h in range(Hq):
        np.testing.assert_array_equal(out[0, h], v[blk, h, 0])


def test_brute_force_tiny():
    r = np.random.Generator(np.random.PCG64(41))
    N, Hq, Hkv, d, B = 3, 4, 2, 3, 2
    ctx = [5, 3, 6]
    qlen = [2, 3, 1]
    k, v, tables = paged_case(r, N, Hq, Hkv, d, B, ctx)
    qs = np.concatenate([[0], np.cumsum(qlen)])
    q = r.standard_normal((qs[-1], Hq, d))
    got = decode_multi_ref(q, k, v, tables, ctx, qs, 0.8)
    g = Hq // Hkv
    for b in range(N):
        for i in range(qlen[b]):
            lim = ctx[b] - qlen[b] + i
            for h in range(Hq):
                s = []
                for t in range(lim + 1):
                    blk, off = tables[b][t // B], t % B
                    s.append(0.8 * sum(q[qs[b] + i, h, j] * k[blk, h // g, off, j] for j in range(d)))
                mx = max(s)
                w = [np.exp(x - mx) for x in s]
                tot = sum(w)
                for j in range(d):
                    want = sum(w[t] / tot * v[tables[b][t // B], h // g, t % B, j] for t in range(lim + 1))
                    assert abs(got[qs[b] + i, h, j] - want) < 1e-12


def test_gqa_equals_mha_with_repeated_kv_heads():
    r = np.random.Generator(np.random.PCG64(51))
    N, Hq, Hkv, d, B = 2, 8, 2, 8, 4
    ctx, qlen = [9, 6], [4, 2]
    k, v, tables = paged_case(r, N, Hq, Hkv, d, B, ctx)
    qs = np.concatenate([[0], np.cumsum(qlen)])
    q = r.standard_normal((qs[-1], Hq, d))
    a = decode_multi_ref(q, k, v, tables, ctx, qs, 0.3)
    km = np.repeat(k, Hq // Hkv, axis=1)
    vm = np.repeat(v, Hq // Hkv, axis=1)
    b = decode_multi_ref(q, km, vm, tables, ctx, qs, 0.3)
    np.testing.assert_array_equal(a, b)


def test_planted_off_by_one_in_the_limit_is_caught():
    # a limit of ctx - q_len + i - 1 (one key short) fails the causal pin
    r = np.random.Generator(np.random.PCG64(61))
    Hq, Hkv, d, ctx, n = 2, 1, 4, 7, 3
    k_seq = r.standard_normal((ctx, Hkv, d))
    v_seq = r.standard_normal((ctx, Hkv, d))
    q_all = r.standard_normal((ctx, Hq, d))
    dense = causal_dense_ref(q_all, k_seq, v_seq, 1.0)
    from oracle.attention import softmax_weights
    wrong = np.array([[softmax_weights(q_all[i, h], k_seq[:i, 0], 1.0) @ v_seq[:i, 0] for h in range(Hq)]
                      for i in range(ctx - n, ctx)])
    assert np.abs(wrong - dense[ctx - n:]).max() > 1e-3
