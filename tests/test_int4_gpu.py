"""The 4-bit cache on the GPU: the quantising append is byte-exact against the
oracle's quantiser; decode over random 4-bit pools matches the fp64 oracle on
the decoded values; whole-block copies are byte-exact."""

import numpy as np
import pytest
import torch

from oracle.attention import decode_ref
from oracle.int4 import append_int4_ref, dequantize_rows, dequantized_pools, split_piece
from tests.gpu_util import assert_close, dev_case, need_gpu
from workloads import CONFIGS, DecodeConfig, make_decode_case, make_int4_pool, make_values

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()


def pa():
    import paged_kv_cache_254_gb300 as m
    return m


def flat(pool):
    NB, Hkv = pool.shape[0], pool.shape[1]
    return pool.reshape(NB, Hkv, -1).cpu().numpy()


@pytest.mark.parametrize("B", [16, 32])
@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_append_is_byte_exact(B, dtype):
    NB, Hkv, d, T = 12, 3, 128, 40
    g = torch.Generator(device="cuda").manual_seed(B)
    pool = torch.randint(0, 256, (NB, Hkv, B, d + 8), generator=g, device="cuda", dtype=torch.int32).to(torch.uint8)
    kn = make_values((T, Hkv, d), dtype, g, "cuda") * 3
    vn = make_values((T, Hkv, d), dtype, g, "cuda")
    kn[0, 0] = 0                                         # a zero row: scale 0, codes 0
    r = np.random.Generator(np.random.PCG64(B + 1))
    slots = r.permutation(NB * B)[:T].astype(np.int64)
    slots[3] = -1                                        # skipped
    want = append_int4_ref(flat(pool), kn.float().cpu().numpy(), vn.float().cpu().numpy(), slots, B)
    pa().pa_append_kv_int4(kn, vn, torch.from_numpy(slots).cuda(), pool)
    got = flat(pool)
    assert (got == want).all(), f"{int((got != want).sum())} bytes differ"


def int4_case(ctx, Hq, Hkv, B, dtype, seed):
    cfg = DecodeConfig(name="int4", num_seqs=len(ctx), num_q_heads=Hq, num_kv_heads=Hkv, head_dim=128,
                       block_size=B, dtype=dtype, seed=seed, ctx_fixed=tuple(ctx), pool_factor=1.3)
    case = make_decode_case(cfg, device="cuda", values=False)
    g = torch.Generator(device="cuda").manual_seed(seed)
    case.q = make_values((len(ctx), Hq, 128), dtype, g, "cuda")
    pool = make_int4_pool(case.num_blocks, Hkv, B, 128, g, "cuda")
    return case, pool


def decode(case, pool, **kw):
    bt, cl = dev_case(case)
    return pa().pa_decode_int4(case.q, pool, bt, cl, case.scale, **kw)


EDGE = [1, 2, 15, 16, 17, 31, 32, 33, 48, 100, 513]


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("B", [16, 32])
@pytest.mark.parametrize("g", [1, 4, 8, 16])
def test_decode_matches_oracle(dtype, B, g):
    Hkv = 2
    case, pool = int4_case(EDGE, Hkv * g, Hkv, B, dtype, seed=100 + B + g)
    kf, vf = dequantized_pools(flat(pool), B, 128)
    want = decode_ref(case.q, kf, vf, case.block_tables, case.context_lens, case.scale)
    assert_close(decode(case, pool), want, what=f"int4 {dtype} B{B} g{g}")


def test_long_contexts_and_splits():
    ctx = [30000, 5, 12000, 800]
    case, pool = int4_case(ctx, 8, 1, 16, "bf16", seed=7)
    kf, vf = dequantized_pools(flat(pool), 16, 128)
    want = decode_ref(case.q, kf, vf, case.block_tables, case.context_lens, case.scale)
    assert_close(decode(case, pool), want, what="long int4")


def test_copy_blocks_is_byte_exact():
    NB, Hkv, B = 16, 4, 16
    g = torch.Generator(device="cuda").manual_seed(3)
    pool = make_int4_pool(NB, Hkv, B, 128, g, "cuda")
    before = pool.clone()
    pairs = torch.tensor([[1, 9], [4, 2], [7, 7]], dtype=torch.int32, device="cuda")
    pa().pa_copy_blocks_int4(pairs, pool)
    want = before.clone()
    want[9] = before[1]
    want[2] = before[4]
    assert torch.equal(pool, want)


def test_full_size_batch_sampled():
    # the 70B-shaped batch over a 4-bit pool, checked on sampled sequences
    cfg = CONFIGS["llama3_70b_b256"]
    case = make_decode_case(cfg, device="cuda", values=False)
    g = torch.Generator(device="cuda").manual_seed(5)
    case.q = make_values((cfg.num_seqs, cfg.num_q_heads, 128), cfg.dtype, g, "cuda")
    pool = make_int4_pool(case.num_blocks, cfg.num_kv_heads, cfg.block_size, 128, g, "cuda")
    out = decode(case, pool)
    assert torch.isfinite(out.float()).all()
    seqs = [0, 77, 255]
    B = cfg.block_size
    for s in seqs:
        nb = -(-int(case.context_lens[s]) // B)
        ids = case.block_tables[s, :nb]
        sub = pool[torch.from_numpy(ids.astype(np.int64)).cuda()]
        kf, vf = dequantized_pools(flat(sub), B, 128)
        want = decode_ref(case.q[s:s + 1], kf, vf, np.arange(nb)[None, :], case.context_lens[s:s + 1], case.scale)
        assert_close(out[s:s + 1], want, what=f"sequence {s}")


def test_long_context_mha_full_size_sampled():
    # 32 sequences x 32,768 tokens x 64 KV heads over a 4-bit pool (9.1 GB),
    # the launch the bench times; sampled (sequence, head) rows checked
    cfg = CONFIGS["long_mha_32k"]
    case = make_decode_case(cfg, device="cuda", values=False)
    g = torch.Generator(device="cuda").manual_seed(31)
    case.q = make_values((cfg.num_seqs, cfg.num_q_heads, 128), cfg.dtype, g, "cuda")
    pool = make_int4_pool(case.num_blocks, cfg.num_kv_heads, cfg.block_size, 128, g, "cuda")
    out = decode(case, pool)
    assert torch.isfinite(out.float()).all()
    B = cfg.block_size
    for s, h in ((0, 0), (13, 37), (31, 63)):
        nb = -(-int(case.context_lens[s]) // B)
        ids = torch.from_numpy(case.block_tables[s, :nb].astype(np.int64)).cuda()
        sub = pool[ids][:, h:h + 1].contiguous()                 # this head's pieces only
        kf, vf = dequantized_pools(flat(sub), B, 128)
        want = decode_ref(case.q[s:s + 1, h:h + 1], kf, vf, np.arange(nb)[None, :], case.context_lens[s:s + 1],
                          case.scale)
        assert_close(out[s:s + 1, h:h + 1], want, what=f"32K MHA sequence {s} head {h}")
    del case, pool
    torch.cuda.empty_cache()


def test_dequantized_values_round_trip_through_append():
    # appended rows decode (oracle side) to code * scale of the pages' rule
    from oracle.int4 import quantize_rows
    NB, Hkv, B, d = 4, 2, 16, 128
    pool = pa().int4_pool(NB, Hkv, B, d)
    g = torch.Generator(device="cuda").manual_seed(9)
    kn = make_values((2, Hkv, d), "bf16", g, "cuda")
    vn = make_values((2, Hkv, d), "bf16", g, "cuda")
    pa().pa_append_kv_int4(kn, vn, torch.tensor([5, 40], dtype=torch.int64, device="cuda"), pool)
    K, V, ks, vs = split_piece(flat(pool)[40 // B, 1], B, d)
    kq, ksc = quantize_rows(kn[1, 1].float().cpu().numpy())
    np.testing.assert_array_equal(dequantize_rows(K[40 % B], ks[40 % B]), dequantize_rows(kq, ksc))


@pytest.mark.parametrize("B", [16, 32])
def test_masked_slots_with_non_finite_scales(B):
    # slots past a context hold scales that are NaN or inf; the kernel must
    # give them no weight whether the partial stage is in its first or
    # second 16-token half
    from oracle.int4 import _offsets
    ctx = [1, 15, 17, 31, 33, 100, 250]
    case, pool = int4_case(ctx, 16, 2, B, "bf16", seed=60 + B)
    kf, vf = dequantized_pools(flat(pool), B, 128)
    want = decode_ref(case.q, kf, vf, case.block_tables, case.context_lens, case.scale)
    _, _, ks, vs = _offsets(B, 128)
    bad = np.array([np.nan, np.inf, -np.inf], dtype=np.float32).view(np.uint8).reshape(3, 4)
    raw = pool.view(pool.shape[0], pool.shape[1], -1)
    for s, c in enumerate(ctx):
        blk = int(case.block_tables[s, (c - 1) // B])
        for off in range(c - ((c - 1) // B) * B, B):
            for base in (ks, vs):
                v = torch.from_numpy(bad[(s + off + base) % 3].copy()).cuda()
                raw[blk, :, base + 4 * off:base + 4 * off + 4] = v
    got = decode(case, pool)
    assert torch.isfinite(got.float()).all()
    assert_close(got, want, what=f"non-finite masked scales B{B}")


# ---- peaked softmaxes over the 4-bit cache ----
def grow_k_scales(case, pool, growth):
    """Multiply the K scale of every sequence's cached token t by
    1 + growth * (t + 1) / ctx, so later keys score higher (the running
    maximum keeps rising)."""
    B = pool.shape[2]
    raw = pool.view(pool.shape[0], pool.shape[1], -1)
    ks = B * 128                                          # K scales follow the K and V codes
    for s, n in enumerate(case.context_lens):
        n = int(n)
        nb = -(-n // B)
        ids = torch.from_numpy(case.block_tables[s, :nb].astype(np.int64)).cuda()
        sc = raw[ids, :, ks:ks + 4 * B].contiguous().view(torch.float32)          # [nb, Hkv, B]
        t = torch.arange(nb * B, device="cuda", dtype=torch.float32).reshape(nb, 1, B)
        sc = sc * (1.0 + growth * (t + 1.0) / n)
        raw[ids, :, ks:ks + 4 * B] = sc.contiguous().view(torch.uint8).view(nb, raw.shape[1], 4 * B)


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("B,g", [(16, 8), (32, 16), (16, 1)])
@pytest.mark.parametrize("q_mult,growth", [(8.0, 0.0), (32.0, 0.0), (2.0, 6.0)])
def test_peaked_softmax(dtype, B, g, q_mult, growth):
    ctx = [3000, 17, 2000, 1, 777, 33, 1500]
    Hkv = 2
    case, pool = int4_case(ctx, Hkv * g, Hkv, B, dtype, seed=400 + B + g)
    case.q.mul_(q_mult)
    if growth:
        grow_k_scales(case, pool, growth)
    kf, vf = dequantized_pools(flat(pool), B, 128)
    want = decode_ref(case.q, kf, vf, case.block_tables, case.context_lens, case.scale)
    assert_close(decode(case, pool), want, what=f"int4 peaked {dtype} B{B} g{g} x{q_mult} +{growth}")
