"""Pins for the fp64 attention oracle: each check ties it to something other
than itself (brute force, closed forms, the un-paged layout, invariants)."""

import json
import math
import os

import numpy as np
import pytest
import scipy.special
import torch

from oracle import sizes
from oracle.attention import (decode_ref, gather_sequence, lse_merge_ref, partial_ref,
                              physical_location, softmax_weights, unpaged_ref)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rng(seed):
    return np.random.Generator(np.random.PCG64(seed))


def build_paged(Kc, Vc, table, num_blocks, B):
    """Lay contiguous caches [ctx, Hkv, d] into a pool [NB, Hkv, B, d] by
    reshaping whole blocks (no per-token index arithmetic), padding the last
    block with NaN so any read past the context poisons the result."""
    ctx, Hkv, d = Kc.shape
    nblk = -(-ctx // B)
    pad = nblk * B - ctx
    kp = np.full((num_blocks, Hkv, B, d), np.nan)
    vp = np.full((num_blocks, Hkv, B, d), np.nan)
    Kb = np.concatenate([Kc, np.full((pad, Hkv, d), np.nan)]).reshape(nblk, B, Hkv, d)
    Vb = np.concatenate([Vc, np.full((pad, Hkv, d), np.nan)]).reshape(nblk, B, Hkv, d)
    kp[table[:nblk]] = Kb.transpose(0, 2, 1, 3)
    vp[table[:nblk]] = Vb.transpose(0, 2, 1, 3)
    return kp, vp


def random_case(seed, ctx, Hq=4, Hkv=2, d=8, B=4, extra_blocks=5):
    r = _rng(seed)
    nblk = -(-ctx // B)
    NB = nblk + extra_blocks
    table = r.permutation(NB)[:nblk]
    Kc = r.standard_normal((ctx, Hkv, d))
    Vc = r.standard_normal((ctx, Hkv, d))
    q = r.standard_normal((Hq, d))
    kp, vp = build_paged(Kc, Vc, table, NB, B)
    row = np.full(nblk + 3, NB + 100)          # unused entries out of range
    row[:nblk] = table
    return q, Kc, Vc, kp, vp, row


def brute_force(q, Kc, Vc, scale):
    """Pure-Python loops with math.exp, one query head at a time."""
    Hq, d = q.shape
    ctx, Hkv, _ = Kc.shape
    g = Hq // Hkv
    out = [[0.0] * d for _ in range(Hq)]
    for h in range(Hq):
        kh = h // g
        s = [scale * sum(q[h][i] * Kc[t][kh][i] for i in range(d)) for t in range(ctx)]
        m = max(s)
        e = [math.exp(x - m) for x in s]
        z = sum(e)
        for i in range(d):
            out[h][i] = sum(e[t] * Vc[t][kh][i] for t in range(ctx)) / z
    return np.array(out)


def one_seq(q, kp, vp, row, ctx, scale):
    return decode_ref(q[None], kp, vp, row[None], np.array([ctx]), scale)[0]


@pytest.mark.parametrize("ctx", [1, 3, 4, 5, 8, 9, 17])
def test_matches_brute_force(ctx):
    q, Kc, Vc, kp, vp, row = random_case(10 + ctx, ctx)
    got = one_seq(q, kp, vp, row, ctx, 0.35)
    np.testing.assert_allclose(got, brute_force(q, Kc, Vc, 0.35), rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("ctx,B", [(1, 16), (15, 16), (16, 16), (17, 16), (32, 16), (100, 16),
                                   (31, 32), (33, 32), (200, 32)])
def test_paged_equals_unpaged(ctx, B):
    q, Kc, Vc, kp, vp, row = random_case(ctx * 7 + B, ctx, Hq=8, Hkv=2, d=16, B=B)
    got = one_seq(q, kp, vp, row, ctx, 0.25)
    np.testing.assert_allclose(got, unpaged_ref(q, Kc, Vc, 0.25), rtol=1e-12, atol=1e-13)
    assert np.isfinite(got).all()


def test_physical_location_formula():
    # Block table formula: logical block i = floor(t / B), offset j = t mod B.
    row = [7, 3, 11]
    assert physical_location(row, 0, 16) == (7, 0)
    assert physical_location(row, 15, 16) == (7, 15)
    assert physical_location(row, 16, 16) == (3, 0)
    assert physical_location(row, 37, 16) == (11, 5)


def test_gather_returns_contiguous_rows():
    q, Kc, Vc, kp, vp, row = random_case(3, 23, B=4)
    for kh in range(2):
        K, V = gather_sequence(kp, vp, row, 23, kh, 4)
        np.testing.assert_array_equal(K, Kc[:, kh])
        np.testing.assert_array_equal(V, Vc[:, kh])


def test_single_token_returns_its_value_exactly():
    q, Kc, Vc, kp, vp, row = random_case(5, 1)
    got = one_seq(q, kp, vp, row, 1, 0.5)
    for h in range(4):
        np.testing.assert_array_equal(got[h], Vc[0, h // 2])


def test_zero_query_is_mean_of_values():
    q, Kc, Vc, kp, vp, row = random_case(6, 29)
    got = one_seq(np.zeros_like(q), kp, vp, row, 29, 0.5)
    for h in range(4):
        np.testing.assert_allclose(got[h], Vc[:, h // 2].mean(axis=0), rtol=1e-13, atol=1e-14)


def test_equal_keys_is_mean_of_values():
    q, Kc, Vc, kp, vp, row = random_case(7, 13)
    Kc[:] = Kc[0]
    kp, vp = build_paged(Kc, Vc, row[:4], kp.shape[0], 4)
    got = one_seq(q, kp, vp, row, 13, 0.5)
    for h in range(4):
        np.testing.assert_allclose(got[h], Vc[:, h // 2].mean(axis=0), rtol=1e-13, atol=1e-14)


def test_dominant_score_selects_its_value():
    q, Kc, Vc, kp, vp, row = random_case(8, 21, Hq=2, Hkv=1, d=8)
    q[:] = 0.0
    q[:, 0] = 1.0
    Kc[:] = 0.0
    Kc[11, 0, 0] = 1000.0          # one score 1e3 above every other
    kp, vp = build_paged(Kc, Vc, row[:6], kp.shape[0], 4)
    got = one_seq(q, kp, vp, row, 21, 1.0)
    for h in range(2):
        np.testing.assert_allclose(got[h], Vc[11, 0], rtol=0, atol=1e-300)


def test_weights_sum_to_one_and_match_scipy():
    r = _rng(9)
    K = r.standard_normal((57, 16))
    qv = r.standard_normal(16)
    p = softmax_weights(qv, K, 0.7)
    assert abs(p.sum() - 1.0) < 1e-14
    np.testing.assert_allclose(p, scipy.special.softmax(0.7 * K @ qv), rtol=1e-13)


def test_scale_folds_into_query():
    q, Kc, Vc, kp, vp, row = random_case(12, 19)
    a = one_seq(q, kp, vp, row, 19, 0.5)
    b = one_seq(q * 0.5, kp, vp, row, 19, 1.0)
    np.testing.assert_allclose(a, b, rtol=1e-13, atol=1e-14)


def test_invariant_under_physical_permutation():
    r = _rng(13)
    N, Hq, Hkv, d, B, NB = 3, 4, 2, 8, 4, 40
    ctx = np.array([9, 17, 4])
    kp = r.standard_normal((NB, Hkv, B, d))
    vp = r.standard_normal((NB, Hkv, B, d))
    q = r.standard_normal((N, Hq, d))
    tables = np.full((N, 6), -1)
    ids = r.permutation(NB)
    pos = 0
    for s in range(N):
        k = -(-ctx[s] // B)
        tables[s, :k] = ids[pos:pos + k]
        pos += k
    base = decode_ref(q, kp, vp, tables, ctx, 0.3)
    for trial in range(3):
        relabel = r.permutation(NB)              # block b moves to relabel[b]
        kp2 = np.empty_like(kp)
        vp2 = np.empty_like(vp)
        kp2[relabel] = kp
        vp2[relabel] = vp
        t2 = np.where(tables >= 0, relabel[np.maximum(tables, 0)], -1)
        np.testing.assert_array_equal(decode_ref(q, kp2, vp2, t2, ctx, 0.3), base)


def test_gqa_equals_mha_with_repeated_kv_heads():
    r = _rng(14)
    ctx, Hq, Hkv, d, B = 23, 8, 2, 8, 4
    g = Hq // Hkv
    Kc = r.standard_normal((ctx, Hkv, d))
    Vc = r.standard_normal((ctx, Hkv, d))
    q = r.standard_normal((Hq, d))
    table = r.permutation(12)[:6]
    kp, vp = build_paged(Kc, Vc, table, 12, B)
    gqa = one_seq(q, kp, vp, table, ctx, 0.4)
    Kr = np.repeat(Kc, g, axis=1)
    Vr = np.repeat(Vc, g, axis=1)
    kp2, vp2 = build_paged(Kr, Vr, table, 12, B)
    mha = one_seq(q, kp2, vp2, table, ctx, 0.4)
    np.testing.assert_array_equal(gqa, mha)


@pytest.mark.parametrize("cuts", [[0, 7, 31], [0, 1, 2, 31], [0, 16, 17, 30, 31], [0, 31]])
def test_partitions_merge_to_one_pass(cuts):
    r = _rng(15)
    K = r.standard_normal((31, 16)) * 3
    V = r.standard_normal((31, 16))
    qv = r.standard_normal(16)
    parts = [partial_ref(qv, K, V, 0.5, lo, hi) for lo, hi in zip(cuts[:-1], cuts[1:])]
    whole = softmax_weights(qv, K, 0.5) @ V
    np.testing.assert_allclose(lse_merge_ref(parts), whole, rtol=1e-13, atol=1e-14)


def test_empty_context_gives_zero_row():
    q, Kc, Vc, kp, vp, row = random_case(16, 5)
    out = decode_ref(q[None], kp, vp, row[None], np.array([0]), 0.5)[0]
    np.testing.assert_array_equal(out, 0.0)


def test_rows_subset_matches_full_and_reads_torch_pools():
    r = _rng(17)
    kp = torch.from_numpy(r.standard_normal((20, 2, 4, 8))).to(torch.bfloat16)
    vp = torch.from_numpy(r.standard_normal((20, 2, 4, 8))).to(torch.bfloat16)
    q = torch.from_numpy(r.standard_normal((2, 4, 8))).to(torch.bfloat16)
    tables = np.array([[3, 9, 1, -1], [0, 12, 7, 5]])
    ctx = np.array([10, 16])
    full = decode_ref(q, kp, vp, tables, ctx, 0.3)
    part = decode_ref(q, kp, vp, tables, ctx, 0.3, rows=[(1, 2), (0, 3)])
    np.testing.assert_array_equal(part[1, 2], full[1, 2])
    np.testing.assert_array_equal(part[0, 3], full[0, 3])
    assert np.isnan(part[0, 0]).all()
    # bf16 widened exactly: same answer as from the fp64 copy of the pools
    full64 = decode_ref(q.double().numpy(), kp.double().numpy(), vp.double().numpy(), tables, ctx, 0.3)
    np.testing.assert_array_equal(full, full64)


# -- pages' worked numbers ---------------------------------------------------

def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


@pytest.mark.parametrize("case", _golden("kv_sizes.json")["cases"], ids=lambda c: c["name"])
def test_kv_sizes_match_pages(case):
    got = getattr(sizes, case["fn"])(**case["args"])
    assert abs(got - case["expected"]) <= case["rel_tol"] * case["expected"]
    if "exact" in case:
        assert got == case["exact"]


def test_gqa_saves_seven_eighths_and_fp8_halves():
    # ontq section 6: one KV head per 8 query heads shrinks KV by 87.5%;
    # 8-bit KV halves it.
    mha = sizes.kv_bytes_per_token(80, 64, 128, 2)
    assert 1 - sizes.kv_bytes_per_token(80, 8, 128, 2) / mha == 0.875
    assert sizes.kv_bytes_per_token(80, 64, 128, 1) / mha == 0.5


def test_on_demand_waste_below_one_block():
    # thewebvale intro: paging keeps fragmentation under 4%; with on-demand
    # allocation a sequence wastes fewer than B slots in its last block.
    r = _rng(18)
    lens = r.integers(1024, 8192, size=256, endpoint=True)
    waste = sum(sizes.wasted_slots(int(n), 16) for n in lens)
    assert all(sizes.wasted_slots(int(n), 16) < 16 for n in lens)
    assert waste / (waste + lens.sum()) < 0.04


def _shared_prefix_case(seed, B=4, groups=((0, 3, 2), (3, 5, 1)), tail_max=9, Hq=4, Hkv=2, d=8):
    """Sequences grouped as (start, end, shared full blocks); members copy the
    first member's leading table entries, then own blocks.  One extra
    sequence sits outside every group."""
    r = _rng(seed)
    N = max(e for _, e, _ in groups) + 1
    ctx = np.zeros(N, dtype=np.int64)
    tables = np.full((N, 12), -1)
    nxt = iter(r.permutation(200))
    for s0, s1, p in groups:
        shared = [next(nxt) for _ in range(p)]
        for s in range(s0, s1):
            ctx[s] = p * B + int(r.integers(0, tail_max))
            own = [next(nxt) for _ in range(-(-ctx[s] // B) - p)]
            tables[s, :len(shared) + len(own)] = shared + own
    ctx[N - 1] = 13
    tables[N - 1, :4] = [next(nxt) for _ in range(4)]
    kp = r.standard_normal((200, Hkv, B, d))
    vp = r.standard_normal((200, Hkv, B, d))
    q = r.standard_normal((N, Hq, d))
    starts = [g[0] for g in groups] + [groups[-1][1]]
    return q, kp, vp, tables, ctx, starts, [g[2] for g in groups]


@pytest.mark.parametrize("seed", [20, 22, 23])
def test_shared_prefix_split_equals_plain_decode(seed):
    from oracle.attention import check_prefix_groups, decode_shared_prefix_ref
    q, kp, vp, tables, ctx, starts, pre = _shared_prefix_case(seed)
    assert check_prefix_groups(tables, ctx, starts, pre, 4)
    a = decode_shared_prefix_ref(q, kp, vp, tables, ctx, 0.3, starts, pre)
    b = decode_ref(q, kp, vp, tables, ctx, 0.3)
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-13)


def test_shared_prefix_reads_the_first_members_table():
    # If a member's table disagrees inside the shared prefix the check fails,
    # and the prefix-aware form follows the group's first member.
    from oracle.attention import check_prefix_groups, decode_shared_prefix_ref
    q, kp, vp, tables, ctx, starts, pre = _shared_prefix_case(21)
    bad = tables.copy()
    bad[1, 0] = 199
    assert not check_prefix_groups(bad, ctx, starts, pre, 4)
    a = decode_shared_prefix_ref(q, kp, vp, bad, ctx, 0.3, starts, pre)
    b = decode_ref(q, kp, vp, tables, ctx, 0.3)
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-13)
    short = ctx.copy()
    short[3] = 2                                   # shorter than its group's shared block
    assert not check_prefix_groups(tables, short, starts, pre, 4)
