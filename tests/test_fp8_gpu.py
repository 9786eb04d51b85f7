"""8-bit (FP8) KV cache: the quantising append is bit-exact against the
oracle's encoder; decode matches the oracle's attention over the dequantised
cache; block copies are byte-exact."""

import numpy as np
import pytest
import torch

from oracle.attention import decode_ref
from oracle.fp8 import append_fp8_ref, dequantized_pools
from oracle.kv_ops import copy_ref
from tests.gpu_util import assert_close, need_gpu, plant_key
from workloads import CONFIGS, DecodeConfig, make_codes, make_decode_case, make_values

pytestmark = pytest.mark.gpu

BELOW = {"e4m3": 0x50, "e5m2": 0x48}   # code magnitudes below ~8 and ~4


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()


def pa():
    import paged_kv_cache_254_gb300 as m
    return m


def u8(t):
    return t.detach().cpu().numpy().copy()


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("B", [16, 32])
def test_append_quantizes_bit_exactly(fmt, dtype, B):
    NB, Hkv, d, T = 30, 4, 128, 200
    g = torch.Generator(device="cuda").manual_seed(1)
    kv = make_codes((NB, Hkv, 2, B, d), g, "cuda")
    kn = make_values((T, Hkv, d), dtype, g, "cuda") * 3
    vn = make_values((T, Hkv, d), dtype, g, "cuda")
    kn[0, 0, :4] = torch.tensor([1e4, -1e4, 1e-7, 0.0])         # saturation and underflow
    r = np.random.Generator(np.random.PCG64(2))
    slots = r.permutation(NB * B)[:T].astype(np.int64)
    slots[::9] = -1
    want = append_fp8_ref(u8(kv), kn.float().cpu().numpy(), vn.float().cpu().numpy(), slots, B, 0.25, 0.125, fmt)
    pa().pa_append_kv_fp8(kn, vn, torch.from_numpy(slots).cuda(), kv, 0.25, 0.125, kv_format=fmt)
    torch.cuda.synchronize()
    assert np.array_equal(u8(kv).reshape(want.shape), want)


def fp8_case(ctx, Hq, Hkv, B, dtype, fmt, seed):
    cfg = DecodeConfig(name="fp8", num_seqs=len(ctx), num_q_heads=Hq, num_kv_heads=Hkv, head_dim=128,
                       block_size=B, dtype=dtype, seed=seed, ctx_fixed=tuple(ctx), pool_factor=1.3)
    case = make_decode_case(cfg, device="cuda", values=False)
    g = torch.Generator(device="cuda").manual_seed(seed)
    q = make_values((len(ctx), Hq, 128), dtype, g, "cuda")
    kv = make_codes((case.num_blocks, Hkv, 2, B, 128), g, "cuda", BELOW[fmt])
    return case, q, kv


def run(case, q, kv, ks, vs, fmt, err=None):
    bt = torch.from_numpy(case.block_tables).cuda()
    cl = torch.from_numpy(case.context_lens).cuda()
    return pa().pa_decode_fp8(q, kv, bt, cl, case.scale, ks, vs, kv_format=fmt, err=err)


def oracle(case, q, kv, ks, vs, fmt, rows=None):
    kf, vf = dequantized_pools(u8(kv), case.cfg.block_size, ks, vs, fmt)
    return decode_ref(q, kf, vf, case.block_tables, case.context_lens, case.scale, rows=rows)


EDGE = [1, 2, 15, 16, 17, 33, 100, 513, 1000, 3001]


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("B", [16, 32])
@pytest.mark.parametrize("g", [1, 4, 8, 16])
def test_decode_matches_oracle(fmt, dtype, B, g):
    case, q, kv = fp8_case(EDGE, 2 * g, 2, B, dtype, fmt, seed=10 + g + B)
    err = pa().new_error_word("cuda")
    out = run(case, q, kv, 0.3, 0.5, fmt, err=err)
    assert pa().pa_read_error(err) == 0
    assert_close(out, oracle(case, q, kv, 0.3, 0.5, fmt), what=f"fp8 {fmt} {dtype} B{B} g{g}")


def test_copy_blocks_of_an_8_bit_cache():
    g = torch.Generator(device="cuda").manual_seed(3)
    kv = make_codes((20, 8, 2, 32, 128), g, "cuda")
    pairs = np.array([[2, 9], [2, 10], [5, 19]], dtype=np.int32)
    want, _ = copy_ref(u8(kv), u8(kv), pairs)
    pa().pa_copy_blocks_fp8(torch.from_numpy(pairs).cuda(), kv)
    torch.cuda.synchronize()
    assert np.array_equal(u8(kv), want)


def test_append_then_decode():
    """The newest token of each sequence goes in through the quantising
    append; decode then reads it back from the 8-bit cache."""
    from oracle.kv_ops import slot_of
    case, q, kv = fp8_case([40, 300, 17, 1], 16, 2, 16, "bf16", "e4m3", seed=5)
    g = torch.Generator(device="cuda").manual_seed(6)
    kn = make_values((4, 2, 128), "bf16", g, "cuda")
    vn = make_values((4, 2, 128), "bf16", g, "cuda")
    slots = np.array([slot_of(case.block_tables[s], int(case.context_lens[s]) - 1, 16) for s in range(4)],
                     dtype=np.int64)
    want = append_fp8_ref(u8(kv), kn.float().cpu().numpy(), vn.float().cpu().numpy(), slots, 16, 0.2, 0.4, "e4m3")
    pa().pa_append_kv_fp8(kn, vn, torch.from_numpy(slots).cuda(), kv, 0.2, 0.4)
    out = run(case, q, kv, 0.2, 0.4, "e4m3")
    kf, vf = dequantized_pools(want, 16, 0.2, 0.4, "e4m3")
    assert_close(out, decode_ref(q, kf, vf, case.block_tables, case.context_lens, case.scale), what="append+decode")


def test_llama3_70b_shape_full_size_sampled():
    cfg = CONFIGS["llama3_70b_b256"]
    case = make_decode_case(cfg, device="cuda", values=False)
    g = torch.Generator(device="cuda").manual_seed(cfg.seed)
    q = make_values((cfg.num_seqs, 64, 128), "bf16", g, "cuda")
    kv = make_codes((case.num_blocks, 8, 2, 16, 128), g, "cuda")
    out = run(case, q, kv, 0.25, 0.25, "e4m3")
    assert torch.isfinite(out.float()).all()
    r = np.random.Generator(np.random.PCG64(7))
    rows = sorted({(int(s), int(h)) for s in r.integers(0, cfg.num_seqs, 8) for h in r.integers(0, 64, 2)})
    kf_rows = oracle_rows(case, q, kv, rows)
    assert_close(out, kf_rows, rows=rows, what="fp8 llama3_70b_b256")


def test_long_context_mha_full_size_sampled():
    # 32 sequences x 32,768 tokens x 64 KV heads over an 8-bit pool (17.2 GB),
    # the launch the bench times; sampled (sequence, head) rows checked
    cfg = CONFIGS["long_mha_32k"]
    case = make_decode_case(cfg, device="cuda", values=False)
    g = torch.Generator(device="cuda").manual_seed(33)
    q = make_values((cfg.num_seqs, 64, 128), "bf16", g, "cuda")
    kv = make_codes((case.num_blocks, 64, 2, 16, 128), g, "cuda")
    out = run(case, q, kv, 0.25, 0.25, "e4m3")
    assert torch.isfinite(out.float()).all()
    for s, h in ((0, 0), (13, 37), (31, 63)):
        nb = -(-int(case.context_lens[s]) // 16)
        ids = torch.from_numpy(case.block_tables[s, :nb].astype(np.int64)).cuda()
        sub = kv[ids][:, h:h + 1].contiguous()                   # this head's pieces only
        kf, vf = dequantized_pools(u8(sub), 16, 0.25, 0.25, "e4m3")
        want = decode_ref(q[s:s + 1, h:h + 1], kf, vf, np.arange(nb)[None, :], case.context_lens[s:s + 1],
                          case.scale)
        assert_close(out[s:s + 1, h:h + 1], want, what=f"32K MHA sequence {s} head {h}")
    del case, kv
    torch.cuda.empty_cache()


def oracle_rows(case, q, kv, rows):
    """Dequantise only the blocks the sampled rows read."""
    need = sorted({int(b) for s, _ in rows for b in case.block_tables[s][:-(-int(case.context_lens[s]) // 16)]})
    remap = {b: i for i, b in enumerate(need)}
    idx = torch.tensor(need, device="cuda")
    kf, vf = dequantized_pools(u8(kv.index_select(0, idx)), 16, 0.25, 0.25, "e4m3")
    tables = np.vectorize(lambda b: remap.get(int(b), -1))(case.block_tables)
    return decode_ref(q, kf, vf, tables, case.context_lens, case.scale, rows=rows)


# ---- every finite code, peaked softmaxes, the quantising append at full batch ----
# All finite codes of a format: magnitudes below 0x7F (E4M3: 0x7F is NaN) or
# 0x7C (E5M2: 0x7C is infinity, above it NaN).  The scales map the largest
# code to |k| = 8 and |v| = 4, the range the tolerance is stated for.
FULL = {"e4m3": (0x7F, 448.0), "e5m2": (0x7C, 57344.0)}


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("B,g", [(16, 8), (32, 16), (16, 1)])
def test_decode_over_every_finite_code(fmt, dtype, B, g):
    below, top = FULL[fmt]
    ctx = [1, 17, 100, 1000, 3001, 5000, 33, 777]
    case, q, _ = fp8_case(ctx, 2 * g, 2, B, dtype, fmt, seed=300 + g + B)
    gen = torch.Generator(device="cuda").manual_seed(301 + g)
    kv = make_codes((case.num_blocks, 2, 2, B, 128), gen, "cuda", below)
    ks, vs = 8.0 / top, 4.0 / top
    err = pa().new_error_word("cuda")
    out = run(case, q, kv, ks, vs, fmt, err=err)
    assert pa().pa_read_error(err) == 0
    assert_close(out, oracle(case, q, kv, ks, vs, fmt), what=f"fp8 full range {fmt} {dtype} B{B} g{g}")


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
@pytest.mark.parametrize("q_mult", [8.0, 32.0])
def test_peaked_softmax(fmt, q_mult):
    ctx = [3000, 17, 5000, 4096, 1, 777, 33, 1500]
    case, q, kv = fp8_case(ctx, 64, 8, 16, "bf16", fmt, seed=310)
    q.mul_(q_mult)
    assert_close(run(case, q, kv, 0.3, 0.5, fmt), oracle(case, q, kv, 0.3, 0.5, fmt), what=f"fp8 peaked {fmt} x{q_mult}")


def test_append_then_decode_full_batch():
    """Every sequence of a 256-sequence batch appends its newest token --
    N(0,1) * 3 values, quantised with scales that use the upper codes -- and
    the decode reads it back, with one planted key that dominates."""
    from oracle.kv_ops import slot_of
    r = np.random.Generator(np.random.PCG64(320))
    ctx = [int(c) for c in r.integers(16, 300, size=256, endpoint=True)]
    case, q, kv = fp8_case(ctx, 16, 2, 16, "bf16", "e4m3", seed=321)
    g = torch.Generator(device="cuda").manual_seed(322)
    kn = make_values((256, 2, 128), "bf16", g, "cuda") * 3
    vn = make_values((256, 2, 128), "bf16", g, "cuda") * 3
    slots = np.array([slot_of(case.block_tables[s], ctx[s] - 1, 16) for s in range(256)], dtype=np.int64)
    ks, vs = 0.05, 0.05
    want = append_fp8_ref(u8(kv), kn.float().cpu().numpy(), vn.float().cpu().numpy(), slots, 16, ks, vs, "e4m3")
    assert (want.reshape(-1) & 0x7F).max() > 0x70        # codes far above the random fill's range
    pa().pa_append_kv_fp8(kn, vn, torch.from_numpy(slots).cuda(), kv, ks, vs)
    torch.cuda.synchronize()
    assert np.array_equal(u8(kv).reshape(want.shape), want)
    out = run(case, q, kv, ks, vs, "e4m3")
    kf, vf = dequantized_pools(want, 16, ks, vs, "e4m3")
    assert_close(out, decode_ref(q, kf, vf, case.block_tables, case.context_lens, case.scale),
                 what="append+decode, full batch")


def test_query_beyond_fp16_range_is_flagged():
    case, q, kv = fp8_case([40, 70], 16, 2, 16, "bf16", "e4m3", seed=330)
    q[1, 3, 5] = 1e6                                     # finite in bf16, not in fp16
    err = pa().new_error_word("cuda")
    out = run(case, q, kv, 0.3, 0.5, "e4m3", err=err)
    assert pa().pa_read_error(err) == 4
    assert int(err.item()) == 64                         # PA_DEVERR_Q_RANGE
    assert torch.isfinite(out[0].float()).all()
