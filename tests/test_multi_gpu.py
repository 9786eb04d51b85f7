"""Parity of the multi-token query kernel (a chunk of new tokens per sequence,
causal within it) with the fp64 oracle.

Launches of up to 16 query rows per (sequence, KV head) pair (max_q_len x
group size) run on the mma.sync kernel; these cases stay there unless noted.
Larger ones run on the tcgen05 kernel (tests/test_multi_tc_gpu.py)."""

import numpy as np
import pytest
import torch

from oracle.attention import decode_multi_ref, decode_ref
from tests.gpu_util import assert_close, dev_case, need_gpu, plant_key, sharpen
from workloads import CONFIGS, DecodeConfig, make_decode_case, make_values

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()


def pa():
    import paged_kv_cache_254_gb300 as m
    return m


def multi_case(ctx, qlens, Hq=8, Hkv=2, d=128, B=16, dtype="bf16", seed=3, poison=False):
    cfg = DecodeConfig(name="multi", num_seqs=len(ctx), num_q_heads=Hq, num_kv_heads=Hkv, head_dim=d,
                       block_size=B, dtype=dtype, seed=seed, ctx_fixed=tuple(ctx), pool_factor=1.5)
    case = make_decode_case(cfg, device="cuda", poison_unused=poison)
    qs = np.concatenate([[0], np.cumsum(qlens)]).astype(np.int32)
    gen = torch.Generator(device="cuda").manual_seed(seed + 5)
    q = make_values((int(qs[-1]), Hq, d), dtype, gen, "cuda")
    return case, q, qs


def run(case, q, qs, max_q=None, **kw):
    bt, cl = dev_case(case)
    return pa().pa_decode_multi(q, case.k_pool, case.v_pool, bt, cl, torch.from_numpy(qs).cuda(), case.scale,
                                max_q_len=max_q, **kw)


def oracle(case, q, qs):
    return decode_multi_ref(q, case.k_pool, case.v_pool, case.block_tables, case.context_lens, qs, case.scale)


EDGE = [1, 2, 15, 16, 17, 31, 33, 64, 100, 517]


def chunk_lens(ctx, max_q, rng):
    return [int(rng.integers(0, min(max_q, c) + 1)) for c in ctx]


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("B", [16, 32])
@pytest.mark.parametrize("g,max_q", [(1, 1), (1, 16), (4, 3), (4, 4), (8, 2), (16, 1)])
def test_shapes_and_chunk_lengths(dtype, d, B, g, max_q):
    rng = np.random.Generator(np.random.PCG64(g * 100 + max_q + d + B))
    Hkv = 2
    qlens = chunk_lens(EDGE, max_q, rng)
    qlens[-1] = min(max_q, EDGE[-1])          # at least one full-size chunk
    case, q, qs = multi_case(EDGE, qlens, Hq=Hkv * g, Hkv=Hkv, d=d, B=B, dtype=dtype,
                             seed=7 + g + max_q + d + B)
    got = run(case, q, qs, max_q=max_q)
    assert_close(got, oracle(case, q, qs), what=f"{dtype} d{d} B{B} g{g} max_q {max_q}")


def test_one_token_chunks_match_decode():
    ctx = [5, 64, 300, 1025]
    case, q, qs = multi_case(ctx, [1] * 4, Hq=16, Hkv=2)
    got = run(case, q, qs)
    want = decode_ref(q, case.k_pool, case.v_pool, case.block_tables, case.context_lens, case.scale)
    assert_close(got, want, what="q_len 1")
    bt, cl = dev_case(case)
    dec = pa().pa_decode(q, case.k_pool, case.v_pool, bt, cl, case.scale)
    assert_close(dec, want, what="pa_decode on the same rows")


def test_prefill_chunks_from_empty_and_poisoned_slots():
    # the first chunk of every prompt (ctx == q_len): token 0 sees only key 0;
    # unused slots and table entries are NaN / out of range
    ctx = [1, 2, 5, 8, 13, 16]
    case, q, qs = multi_case(ctx, ctx, Hq=8, Hkv=8, B=16, poison=True)
    got = run(case, q, qs, max_q=16)
    ref = oracle(case, q, qs)
    assert_close(got, ref, what="prefill chunks")
    # token 0 of each chunk equals v_0 up to the output rounding
    for b, r0 in enumerate(qs[:-1]):
        blk = int(case.block_tables[b, 0])
        v0 = case.v_pool[blk, :, 0].float().cpu().numpy()
        np.testing.assert_allclose(got[r0].float().cpu().numpy(), v0, rtol=1e-2, atol=2e-3)


def test_long_contexts_split_across_ctas():
    # long pairs are cut across CTAs: pieces merged by the post-pass
    ctx = [20000, 17, 9000, 33000]
    qlens = [4, 4, 2, 4]
    case, q, qs = multi_case(ctx, qlens, Hq=4, Hkv=1, d=128, B=16, seed=19, poison=True)
    assert_close(run(case, q, qs, max_q=4), oracle(case, q, qs), what="long contexts")


def test_deterministic_and_placement_invariant():
    ctx = [700, 3000, 45, 1200]
    qlens = [3, 4, 1, 4]
    case, q, qs = multi_case(ctx, qlens, Hq=16, Hkv=4, seed=23)
    a = run(case, q, qs, max_q=4)
    b = run(case, q, qs, max_q=4)
    assert torch.equal(a, b)
    # relabel every physical block (same contents at new ids)
    nb = case.num_blocks
    perm = np.random.Generator(np.random.PCG64(1)).permutation(nb)
    k2 = torch.empty_like(case.k_pool)
    v2 = torch.empty_like(case.v_pool)
    pt = torch.from_numpy(perm).cuda()
    k2[pt] = case.k_pool
    v2[pt] = case.v_pool
    tables = np.where(case.block_tables >= 0, perm[np.clip(case.block_tables, 0, nb - 1)], -1).astype(np.int32)
    cl = torch.from_numpy(case.context_lens).cuda()
    c = pa().pa_decode_multi(q, k2, v2, torch.from_numpy(tables).cuda(), cl, torch.from_numpy(qs).cuda(),
                             case.scale, max_q_len=4)
    assert torch.equal(a, c)


def test_malformed_chunks_poison_their_rows_only():
    ctx = [10, 40, 3, 70]
    qlens = [2, 9, 5, 1]           # with max_q_len 6: seq 1's chunk is too long, seq 2's exceeds its context
    case, q, qs = multi_case(ctx, qlens, Hq=4, Hkv=2, seed=29)
    err = pa().new_error_word("cuda")
    got = run(case, q, qs, max_q=6, err=err)
    assert pa().pa_read_error(err) == 4
    assert int(err.item()) & 2
    g = got.float()
    assert torch.isnan(g[qs[1]:qs[2]]).all()        # chunk longer than max_q_len
    assert torch.isnan(g[qs[2]:qs[3]]).all()        # chunk longer than its context
    # the well-formed sequences 0 and 3, as a batch of their own for the oracle
    keep = list(range(qs[0], qs[1])) + list(range(qs[3], qs[4]))
    sub_qs = np.array([0, qs[1] - qs[0], qs[1] - qs[0] + qs[4] - qs[3]], dtype=np.int32)
    ref = decode_multi_ref(q[keep], case.k_pool, case.v_pool, case.block_tables[[0, 3]],
                           case.context_lens[[0, 3]], sub_qs, case.scale)
    assert_close(got[keep], ref, what="well-formed chunks")


def test_speculative_verify_batch_sampled():
    # the 70B-shaped batch with 2-token chunks (one drafted token + one; 16
    # rows per pair), checked on its first 6 sequences
    cfg = CONFIGS["llama3_70b_b256"]
    case = make_decode_case(cfg, device="cuda", seed=41)
    N = len(case.context_lens)
    qs = (np.arange(N + 1) * 2).astype(np.int32)
    gen = torch.Generator(device="cuda").manual_seed(43)
    q = make_values((2 * N, cfg.num_q_heads, cfg.head_dim), cfg.dtype, gen, "cuda")
    got = run(case, q, qs, max_q=2)
    n = 6
    ref = decode_multi_ref(q[:2 * n], case.k_pool, case.v_pool, case.block_tables[:n], case.context_lens[:n],
                           qs[:n + 1], case.scale)
    assert_close(got[:2 * n], ref, what="70B batch, 2-token chunks")
    assert torch.isfinite(got.float()).all()


def test_host_rejects_unsupported_chunks():
    case, q, qs = multi_case([40], [1], Hq=16, Hkv=1)
    with pytest.raises(pa().PagedAttentionError, match="UNSUPPORTED"):
        run(case, q, qs, max_q=9)                # 9 x 16 rows > 128
    with pytest.raises(pa().PagedAttentionError, match="INVALID"):
        run(case, q, qs, max_q=17)


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("q_mult,k_growth", [(8.0, 0.0), (32.0, 0.0), (2.0, 6.0)])
@pytest.mark.parametrize("g,max_q", [(8, 2), (4, 2), (1, 16)])
def test_peaked_chunks(dtype, q_mult, k_growth, g, max_q):
    # mma.sync kernel (up to 16 query rows per pair) on peaked softmaxes
    ctx = [3000, 17, 2000, 4, 777, 33, 1500]
    rng = np.random.Generator(np.random.PCG64(500 + g + max_q))
    qlens = chunk_lens(ctx, max_q, rng)
    qlens[0] = max_q
    case, q, qs = multi_case(ctx, qlens, Hq=2 * g, Hkv=2, dtype=dtype, seed=501 + g)
    q.mul_(q_mult)
    sharpen(case, 1.0, k_growth)
    assert_close(run(case, q, qs, max_q=max_q), oracle(case, q, qs), what=f"peaked chunks {dtype} g{g} q{max_q}")


def test_dominant_keys_inside_and_before_the_chunk():
    ctx = [2500, 700, 40]
    qlens = [4, 3, 4]
    case, q, qs = multi_case(ctx, qlens, Hq=8, Hkv=2, seed=511)
    # for the first chunk token of sequence 0: a key far before the chunk, and
    # one inside the chunk that only its later tokens see
    plant_key(case, 0, 1000, target=20.0, q=q[qs[0]])
    plant_key(case, 0, 2498, target=35.0, q=q[qs[0] + 3])
    plant_key(case, 1, 698, target=28.0, q=q[qs[1] + 2])
    assert_close(run(case, q, qs, max_q=4), oracle(case, q, qs), what="planted keys, multi-token")
