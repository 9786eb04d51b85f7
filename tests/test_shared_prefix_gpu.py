"""Prefix-aware decode (pa_decode_shared_prefix) against the oracle and
against plain pa_decode, on small shapes with edge cases and on the full
parallel-sampling workload."""

import numpy as np
import pytest
import torch

from oracle.attention import decode_ref, decode_shared_prefix_ref
from oracle.kv_ops import append_ref, bits, copy_ref, slot_of
from tests.gpu_util import ATOL, RTOL, assert_close, from_bits, need_gpu, plant_key
from workloads import SAMPLINGS, make_sampling_case, make_values, sampling_tables

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()


def pa():
    import paged_kv_cache_254_gb300 as m
    return m


def grouped_case(seed, groups, Hq, Hkv, d, B, dtype, solo=(13, 1)):
    """groups: list of (members, shared full blocks, tail lengths or None).
    Members share the group's leading blocks, then own blocks.  `solo`
    sequences follow, outside every group."""
    r = np.random.Generator(np.random.PCG64(seed))
    ctx, rows = [], []
    nb_total = 0
    starts, prefix = [0], []
    for members, p, tails in groups:
        shared = list(range(nb_total, nb_total + p))
        nb_total += p
        for m in range(members):
            t = int(tails[m]) if tails is not None else int(r.integers(0, 3 * B))
            n = p * B + t
            own = -(-n // B) - p
            rows.append(shared + list(range(nb_total, nb_total + own)))
            nb_total += own
            ctx.append(n)
        starts.append(starts[-1] + members)
        prefix.append(p)
    for n in solo:
        k = -(-n // B)
        rows.append(list(range(nb_total, nb_total + k)))
        nb_total += k
        ctx.append(n)
    NB = nb_total + 7
    relabel = r.permutation(NB)                     # scatter blocks through the pool
    MB = max(len(x) for x in rows) + 2
    tables = np.full((len(rows), MB), -1, dtype=np.int32)
    for i, x in enumerate(rows):
        tables[i, :len(x)] = relabel[np.asarray(x, dtype=np.int64)] if x else []
    g = torch.Generator(device="cuda").manual_seed(seed)
    q = make_values((len(rows), Hq, d), dtype, g, "cuda")
    kp = make_values((NB, Hkv, B, d), dtype, g, "cuda")
    vp = make_values((NB, Hkv, B, d), dtype, g, "cuda")
    return q, kp, vp, tables, np.asarray(ctx, dtype=np.int32), np.asarray(starts, np.int32), \
        np.asarray(prefix, np.int32)


def run_sp(q, kp, vp, tables, ctx, starts, prefix, scale, err=None):
    c = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()  # noqa: E731
    return pa().pa_decode_shared_prefix(q, kp, vp, c(tables), c(ctx), c(starts), c(prefix), scale, err=err)


CASES = [
    ("bf16", 128, 16, 4, [(8, 5, None), (1, 3, None), (3, 2, [0, 16, 40])]),
    ("fp16", 64, 32, 8, [(5, 2, None), (2, 4, [0, 1])]),
    ("bf16", 128, 32, 16, [(4, 3, None)]),
    ("bf16", 64, 16, 1, [(20, 6, None)]),
    ("bf16", 128, 16, 8, [(12, 4, None), (6, 1, None)]),   # 96 rows: three row chunks
]


@pytest.mark.parametrize("dtype,d,B,g,groups", CASES)
def test_matches_oracle_and_plain_decode(dtype, d, B, g, groups):
    Hkv = 2
    q, kp, vp, tables, ctx, starts, prefix = grouped_case(d + B + g, groups, Hkv * g, Hkv, d, B, dtype)
    scale = float(np.float32(d ** -0.5))
    err = pa().new_error_word("cuda")
    out = run_sp(q, kp, vp, tables, ctx, starts, prefix, scale, err=err)
    assert pa().pa_read_error(err) == 0
    ref = decode_shared_prefix_ref(q, kp, vp, tables, ctx, scale, starts, prefix)
    assert_close(out, ref, what=f"shared prefix {dtype} d{d} B{B} g{g}")
    plain = pa().pa_decode(q, kp, vp, torch.from_numpy(tables).cuda(), torch.from_numpy(ctx).cuda(), scale)
    a, b = out.double(), plain.double()
    assert ((a - b).abs() <= ATOL + RTOL * b.abs()).all()


def test_no_groups_is_plain_decode():
    q, kp, vp, tables, ctx, _, _ = grouped_case(3, [(3, 2, None)], 8, 2, 128, 16, "bf16")
    out = run_sp(q, kp, vp, tables, ctx, np.zeros(1, np.int32), np.zeros(0, np.int32), 0.088)
    plain = pa().pa_decode(q, kp, vp, torch.from_numpy(tables).cuda(), torch.from_numpy(ctx).cuda(), 0.088)
    assert torch.equal(out, plain)


def test_member_breaking_the_prefix_is_flagged_and_poisoned():
    q, kp, vp, tables, ctx, starts, prefix = grouped_case(5, [(4, 3, None), (3, 2, None)], 8, 2, 128, 16, "bf16")
    bad = tables.copy()
    bad[2, 1] = int(tables[5, 0])                               # a block of another group
    err = pa().new_error_word("cuda")
    out = run_sp(q, kp, vp, bad, ctx, starts, prefix, 0.088, err=err)
    assert int(err.item()) & 32
    assert torch.isnan(out[0:4].float()).all()                  # the whole first group
    ref = decode_ref(q, kp, vp, tables, ctx, 0.088)
    keep = list(range(4, len(ctx)))
    assert_close(out[keep], ref[keep], what="other groups untouched")


def test_malformed_description_falls_back_to_plain_attention():
    q, kp, vp, tables, ctx, starts, prefix = grouped_case(6, [(3, 2, None)], 8, 2, 128, 16, "bf16")
    err = pa().new_error_word("cuda")
    wild = prefix.copy()
    wild[0] = tables.shape[1] + 5                                # more blocks than the table has
    out = run_sp(q, kp, vp, tables, ctx, starts, wild, 0.088, err=err)
    assert int(err.item()) & 32
    assert_close(out, decode_ref(q, kp, vp, tables, ctx, 0.088), what="malformed group")


@pytest.mark.parametrize("cfg_name", ["parallel_sampling", "parallel_sampling_aligned"])
def test_parallel_sampling_full_size(cfg_name):
    """64 prompts x 8 samples: copy-on-write (none when the prompt fills its
    blocks), append, then prefix-aware decode over the full shared blocks."""
    case = make_sampling_case(SAMPLINGS[cfg_name], device="cuda")
    cfg = case.cfg
    B, S = cfg.block_size, cfg.samples
    tables, ctx = sampling_tables(case)
    pairs = np.array([[case.prompt_blocks[i // S][-1], case.private_last[i]]
                      for i in range(len(ctx)) if case.private_last[i] >= 0], dtype=np.int32).reshape(-1, 2)
    slots = np.concatenate([[slot_of(tables[i], t, B) for t in range(cfg.prompt_len, int(ctx[i]))]
                            for i in range(len(ctx))]).astype(np.int64)
    wk, wv = copy_ref(bits(case.k_pool), bits(case.v_pool), pairs)
    wk, wv = append_ref(wk, wv, bits(case.k_new), bits(case.v_new), slots, B)
    pa().pa_copy_blocks(torch.from_numpy(pairs).cuda(), case.k_pool, case.v_pool)
    pa().pa_append_kv(case.k_new, case.v_new, torch.from_numpy(slots).cuda(), case.k_pool, case.v_pool)
    starts = np.arange(0, len(ctx) + 1, S, dtype=np.int32)
    prefix = np.full(cfg.groups, cfg.prompt_len // B, dtype=np.int32)          # the full shared blocks
    err = pa().new_error_word("cuda")
    out = run_sp(case.q, case.k_pool, case.v_pool, tables, ctx, starts, prefix, case.scale, err=err)
    assert pa().pa_read_error(err) == 0
    dt = case.q.dtype
    r = np.random.Generator(np.random.PCG64(9))
    rows = sorted({(int(s), int(h)) for s in r.integers(0, len(ctx), size=12) for h in r.integers(0, 32, size=2)})
    ref = decode_shared_prefix_ref(case.q, from_bits(wk, dt), from_bits(wv, dt), tables, ctx, case.scale,
                                   starts, prefix, rows=rows)
    assert_close(out, ref, rows=rows, what="parallel sampling, prefix-aware")
    plain = pa().pa_decode(case.q, case.k_pool, case.v_pool, torch.from_numpy(tables).cuda(),
                           torch.from_numpy(ctx).cuda(), case.scale)
    a, b = out.double(), plain.double()
    assert ((a - b).abs() <= ATOL + RTOL * b.abs()).all()


@pytest.mark.parametrize("groups,what", [
    # 30 groups x 2 KV heads of 12 shared blocks: each item is cut across
    # several CTA ranges (a few pieces, merged through shared memory)
    ([(4, 12, None)] * 30, "few pieces"),
    # one group with a 400-block prompt: its items span far more CTA ranges
    # than the shared-memory merge holds (the in-order fold)
    ([(4, 400, None)], "many pieces"),
])
def test_prefix_items_split_across_many_ctas(groups, what):
    q, kp, vp, tables, ctx, starts, prefix = grouped_case(77, groups, 8, 2, 128, 16, "bf16", solo=(5,))
    scale = float(np.float32(128 ** -0.5))
    err = pa().new_error_word("cuda")
    out = run_sp(q, kp, vp, tables, ctx, starts, prefix, scale, err=err)
    assert pa().pa_read_error(err) == 0
    r = np.random.Generator(np.random.PCG64(3))
    rows = sorted({(int(s), int(h)) for s in r.integers(0, len(ctx), size=10) for h in r.integers(0, 8, size=2)})
    ref = decode_shared_prefix_ref(q, kp, vp, tables, ctx, scale, starts, prefix, rows=rows)
    assert_close(out, ref, rows=rows, what=f"shared prefix, {what}")
    plain = pa().pa_decode(q, kp, vp, torch.from_numpy(tables).cuda(), torch.from_numpy(ctx).cuda(), scale)
    a, b = out.double(), plain.double()
    assert ((a - b).abs() <= ATOL + RTOL * b.abs()).all()


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("q_mult", [1.0, 8.0])
def test_dominant_keys_in_prefix_and_suffix(dtype, q_mult):
    """One key planted in the shared prefix and others in members' own
    blocks, of different heights, so the prefix state (the carry) and the
    suffix disagree on the running maximum in both directions."""
    from types import SimpleNamespace
    d, B, g = 128, 16, 4
    groups = [(8, 40, [5, 70, 16, 0, 33, 100, 1, 64]), (4, 12, [300, 2, 47, 9])]
    q, kp, vp, tables, ctx, starts, prefix = grouped_case(91, groups, 4 * g, 4, d, B, dtype, solo=(900, 5))
    q.mul_(q_mult)
    scale = float(np.float32(1.0 / np.sqrt(d)))
    c = SimpleNamespace(q=q, k_pool=kp, block_tables=tables, scale=scale)
    plant_key(c, 0, 37, target=18.0)              # in group 0's shared prefix (40 blocks)
    plant_key(c, 8, 12 * B + 200, target=30.0)    # in member 8's own blocks (group 1)
    plant_key(c, 2, 40 * B + 10, target=9.0)      # below group 0's prefix key for its first head
    plant_key(c, 3, 3, target=40.0)               # far above, inside the prefix again
    plant_key(c, 12, 850, target=25.0)            # a sequence outside every group
    err = pa().new_error_word("cuda")
    got = run_sp(q, kp, vp, tables, ctx, starts, prefix, scale, err=err)
    assert pa().pa_read_error(err) == 0
    assert_close(got, decode_ref(q, kp, vp, tables, ctx, scale), what=f"planted keys {dtype} x{q_mult}")
