"""Parity of the tensor-core (tcgen05) multi-token kernel with the fp64 oracle.

Launches whose (sequence, KV head) pairs carry more than 16 query rows
(max_q_len x group size) run on the 128-row tcgen05 kernel; smaller ones on
the mma.sync kernel.  These cases sit above the threshold unless noted."""

import numpy as np
import pytest
import torch

from oracle.attention import decode_multi_ref
from tests.gpu_util import assert_close, dev_case, need_gpu, plant_key, sharpen
from workloads import CONFIGS, DecodeConfig, make_decode_case, make_values

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()


def pa():
    import paged_kv_cache_254_gb300 as m
    return m


def multi_case(ctx, qlens, Hq, Hkv, d=128, B=16, dtype="bf16", seed=3, poison=False):
    cfg = DecodeConfig(name="multi_tc", num_seqs=len(ctx), num_q_heads=Hq, num_kv_heads=Hkv, head_dim=d,
                       block_size=B, dtype=dtype, seed=seed, ctx_fixed=tuple(ctx), pool_factor=1.5)
    case = make_decode_case(cfg, device="cuda", poison_unused=poison)
    qs = np.concatenate([[0], np.cumsum(qlens)]).astype(np.int32)
    gen = torch.Generator(device="cuda").manual_seed(seed + 5)
    q = make_values((int(qs[-1]), Hq, d), dtype, gen, "cuda")
    return case, q, qs


def run(case, q, qs, max_q, **kw):
    bt, cl = dev_case(case)
    return pa().pa_decode_multi(q, case.k_pool, case.v_pool, bt, cl, torch.from_numpy(qs).cuda(), case.scale,
                                max_q_len=max_q, **kw)


def oracle(case, q, qs):
    return decode_multi_ref(q, case.k_pool, case.v_pool, case.block_tables, case.context_lens, qs, case.scale)


EDGE = [1, 2, 15, 16, 17, 31, 33, 63, 64, 65, 100, 129, 517]


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("B", [16, 32])
@pytest.mark.parametrize("g,max_q", [(4, 5), (8, 3), (16, 2), (4, 9), (8, 5), (8, 8), (16, 3), (16, 8), (4, 16)])
def test_ragged_chunks(dtype, d, B, g, max_q):
    rng = np.random.Generator(np.random.PCG64(1000 + 10 * g + max_q + d + B))
    qlens = [int(rng.integers(0, min(max_q, c) + 1)) for c in EDGE]
    qlens[-1] = min(max_q, EDGE[-1])
    qlens[3] = 0                                    # an empty chunk
    case, q, qs = multi_case(EDGE, qlens, Hq=2 * g, Hkv=2, d=d, B=B, dtype=dtype, seed=50 + g + max_q + d + B,
                             poison=True)
    assert_close(run(case, q, qs, max_q), oracle(case, q, qs), what=f"{dtype} d{d} B{B} g{g} max_q {max_q}")


@pytest.mark.parametrize("B", [16, 32])
def test_long_contexts_split_across_ctas(B):
    # pairs far longer than a CTA's share leave partial states for the merge
    ctx = [20000, 17, 9000, 33000, 64, 4097]
    qlens = [8, 8, 3, 8, 1, 6]
    case, q, qs = multi_case(ctx, qlens, Hq=8, Hkv=1, B=B, seed=19 + B, poison=True)
    assert_close(run(case, q, qs, max_q=8), oracle(case, q, qs), what=f"long contexts B{B}")


def test_prefill_chunks_from_empty_cache():
    # the first chunk of each prompt: token 0 sees key 0 alone
    ctx = [1, 2, 5, 8, 13, 16]
    case, q, qs = multi_case(ctx, ctx, Hq=16, Hkv=4, seed=31, poison=True)
    got = run(case, q, qs, max_q=16)
    assert_close(got, oracle(case, q, qs), what="prefill chunks")
    for b, r0 in enumerate(qs[:-1]):
        v0 = case.v_pool[int(case.block_tables[b, 0]), :, 0].float().cpu().numpy()    # [Hkv, d]
        np.testing.assert_allclose(got[r0].float().cpu().numpy(), np.repeat(v0, 4, axis=0), rtol=1e-2, atol=2e-3)


def test_same_answer_as_the_mma_sync_kernel():
    # max_q_len 2 (16 rows) runs the mma.sync kernel, max_q_len 3 the tcgen05
    # one; chunks of at most 2 tokens are valid for both
    ctx = [700, 3000, 45, 1200, 5, 64]
    qlens = [2, 1, 2, 1, 2, 2]
    case, q, qs = multi_case(ctx, qlens, Hq=16, Hkv=2, seed=23, poison=True)
    a = run(case, q, qs, max_q=2)
    b = run(case, q, qs, max_q=3)
    ref = oracle(case, q, qs)
    assert_close(a, ref, what="mma.sync")
    assert_close(b, ref, what="tcgen05")
    np.testing.assert_allclose(a.float().cpu().numpy(), b.float().cpu().numpy(), rtol=1e-2, atol=2e-3)


def test_deterministic_and_placement_invariant():
    ctx = [700, 3000, 45, 1200]
    qlens = [8, 5, 1, 8]
    case, q, qs = multi_case(ctx, qlens, Hq=16, Hkv=2, seed=29)
    a = run(case, q, qs, max_q=8)
    assert torch.equal(a, run(case, q, qs, max_q=8))
    nb = case.num_blocks
    perm = np.random.Generator(np.random.PCG64(2)).permutation(nb)
    k2 = torch.empty_like(case.k_pool)
    v2 = torch.empty_like(case.v_pool)
    pt = torch.from_numpy(perm).cuda()
    k2[pt] = case.k_pool
    v2[pt] = case.v_pool
    tables = np.where(case.block_tables >= 0, perm[np.clip(case.block_tables, 0, nb - 1)], -1).astype(np.int32)
    c = pa().pa_decode_multi(q, k2, v2, torch.from_numpy(tables).cuda(), torch.from_numpy(case.context_lens).cuda(),
                             torch.from_numpy(qs).cuda(), case.scale, max_q_len=8)
    assert torch.equal(a, c)


def test_malformed_chunks_and_bad_block_ids():
    ctx = [10, 40, 3, 70, 300]
    qlens = [2, 9, 5, 1, 6]        # max_q_len 6: seq 1 too long, seq 2 longer than its context
    case, q, qs = multi_case(ctx, qlens, Hq=16, Hkv=2, seed=37)
    tables = case.block_tables.copy()
    tables[4, 7] = case.num_blocks + 5              # a bad block id inside seq 4's context
    err = pa().new_error_word("cuda")
    bt = torch.from_numpy(tables).cuda()
    cl = torch.from_numpy(case.context_lens).cuda()
    got = pa().pa_decode_multi(q, case.k_pool, case.v_pool, bt, cl, torch.from_numpy(qs).cuda(), case.scale,
                               max_q_len=6, err=err)
    word = int(err.item())
    assert word & 1 and word & 2
    g = got.float()
    assert torch.isnan(g[qs[1]:qs[2]]).all()
    assert torch.isnan(g[qs[2]:qs[3]]).all()
    assert torch.isnan(g[qs[4]:qs[5]]).all()
    keep = list(range(qs[0], qs[1])) + list(range(qs[3], qs[4]))
    sub_qs = np.array([0, qs[1] - qs[0], qs[1] - qs[0] + qs[4] - qs[3]], dtype=np.int32)
    ref = decode_multi_ref(q[keep], case.k_pool, case.v_pool, case.block_tables[[0, 3]], case.context_lens[[0, 3]],
                           sub_qs, case.scale)
    assert_close(got[keep], ref, what="well-formed chunks")


def test_large_scores_rescale_lazily():
    # keys that grow along the context push the running maximum up stage after
    # stage, so the output accumulator is rescaled in tensor memory many times
    ctx = [2000, 700]
    case, q, qs = multi_case(ctx, [8, 8], Hq=8, Hkv=1, seed=41)
    B = case.cfg.block_size
    for s, c in enumerate(ctx):
        for t in range(c):
            blk, off = int(case.block_tables[s, t // B]), t % B
            case.k_pool[blk, 0, off] *= 1.0 + 6.0 * t / c
    assert_close(run(case, q, qs, max_q=8), oracle(case, q, qs), what="growing scores")


def test_verify_batch_16_token_chunks_sampled():
    # the 70B-shaped batch with 16-token chunks: 128 query rows per pair
    cfg = CONFIGS["llama3_70b_b256"]
    case = make_decode_case(cfg, device="cuda", seed=43)
    N = len(case.context_lens)
    qs = (np.arange(N + 1) * 16).astype(np.int32)
    gen = torch.Generator(device="cuda").manual_seed(47)
    q = make_values((16 * N, cfg.num_q_heads, cfg.head_dim), cfg.dtype, gen, "cuda")
    got = run(case, q, qs, max_q=16)
    assert torch.isfinite(got.float()).all()
    for s in (0, 101, 255):
        ref = decode_multi_ref(q[16 * s:16 * s + 16], case.k_pool, case.v_pool, case.block_tables[s:s + 1],
                               case.context_lens[s:s + 1], np.array([0, 16], dtype=np.int32), case.scale)
        assert_close(got[16 * s:16 * s + 16], ref, what=f"sequence {s}")


@pytest.mark.parametrize("max_q", [2, 4, 8])  # 16 rows per pair: mma.sync kernel; 32, 64 rows: tcgen05
def test_bad_context_length_poisons_its_rows(max_q):
    ctx = [300, 500, 77, 1000]
    qlens = [max_q, 2, min(3, max_q), max_q]
    case, q, qs = multi_case(ctx, qlens, Hq=16, Hkv=2, seed=53)
    cl = case.context_lens.copy()
    cl[1] = case.block_tables.shape[1] * case.cfg.block_size + 5      # longer than its table can hold
    err = pa().new_error_word("cuda")
    bt = torch.from_numpy(case.block_tables).cuda()
    got = pa().pa_decode_multi(q, case.k_pool, case.v_pool, bt, torch.from_numpy(cl).cuda(),
                               torch.from_numpy(qs).cuda(), case.scale, max_q_len=max_q, err=err)
    assert int(err.item()) & 2
    assert torch.isnan(got[qs[1]:qs[2]].float()).all()
    keep = [i for s in (0, 2, 3) for i in range(qs[s], qs[s + 1])]
    sub = [0, 2, 3]
    sub_qs = np.concatenate([[0], np.cumsum([qlens[s] for s in sub])]).astype(np.int32)
    ref = decode_multi_ref(q[keep], case.k_pool, case.v_pool, case.block_tables[sub], case.context_lens[sub],
                           sub_qs, case.scale)
    assert_close(got[keep], ref, what=f"well-formed sequences, max_q {max_q}")


@pytest.mark.parametrize("q_mult", [8.0, 32.0])
@pytest.mark.parametrize("max_q", [3, 8])         # 24 and 64 query rows per pair
def test_peaked_and_planted_keys_tcgen05(q_mult, max_q):
    # tcgen05 kernel: peaked scores plus keys that dominate late in long split
    # contexts and inside the chunk
    ctx = [3000, 2000, 777, 64]
    qlens = [max_q, min(5, max_q), max_q, max_q]
    case, q, qs = multi_case(ctx, qlens, Hq=16, Hkv=2, seed=521 + max_q)
    q.mul_(q_mult)
    plant_key(case, 0, 2950, target=60.0, q=q[qs[0]])
    plant_key(case, 1, 1998, target=45.0, q=q[qs[1] + min(4, max_q - 1)])
    plant_key(case, 2, 100, target=50.0, q=q[qs[2] + 1])
    assert_close(run(case, q, qs, max_q=max_q), oracle(case, q, qs), what=f"tcgen05 peaked x{q_mult} q{max_q}")


@pytest.mark.parametrize("config,q_len", [("llama3_70b_b256", 3), ("llama3_70b_b256", 4), ("llama3_70b_b256", 8),
                                          ("llama3_8b_b64", 8), ("llama3_8b_b64", 16)])
def test_verify_batch_chunks_sampled(config, q_len):
    # the bench's multi-token batches (q_len new tokens per sequence: 24 to
    # 64 rows per pair), checked on sequences spread over the batch
    cfg = CONFIGS[config]
    case = make_decode_case(cfg, device="cuda", seed=41 + q_len)
    N = len(case.context_lens)
    qs = (np.arange(N + 1) * q_len).astype(np.int32)
    gen = torch.Generator(device="cuda").manual_seed(43 + q_len)
    q = make_values((q_len * N, cfg.num_q_heads, cfg.head_dim), cfg.dtype, gen, "cuda")
    got = run(case, q, qs, max_q=q_len)
    assert torch.isfinite(got.float()).all()
    for s in (0, N // 3, N - 1):
        ref = decode_multi_ref(q[q_len * s:q_len * (s + 1)], case.k_pool, case.v_pool, case.block_tables[s:s + 1],
                               case.context_lens[s:s + 1], np.array([0, q_len], dtype=np.int32), case.scale)
        assert_close(got[q_len * s:q_len * (s + 1)], ref, what=f"{config} {q_len}-token chunks, sequence {s}")
