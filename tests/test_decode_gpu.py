"""Parity of the CUDA paged decode kernel with the fp64 oracle."""

import numpy as np
import pytest
import torch

from oracle.attention import decode_ref
from tests.gpu_util import assert_close, dev_case, need_gpu, plant_key, sharpen
from workloads import CONFIGS, DecodeConfig, make_decode_case

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()


def pa():
    import paged_kv_cache_254_gb300 as m
    return m


def run(case, **kw):
    bt, cl = dev_case(case)
    return pa().pa_decode(case.q, case.k_pool, case.v_pool, bt, cl, case.scale, **kw)


def oracle(case, rows=None):
    return decode_ref(case.q, case.k_pool, case.v_pool, case.block_tables, case.context_lens, case.scale,
                      rows=rows)


def small_cfg(ctx, Hq=8, Hkv=2, d=128, B=16, dtype="bf16", seed=7):
    return DecodeConfig(name="small", num_seqs=len(ctx), num_q_heads=Hq, num_kv_heads=Hkv, head_dim=d,
                        block_size=B, dtype=dtype, seed=seed, ctx_fixed=tuple(ctx), pool_factor=1.5)


def test_tiny_config_full():
    case = make_decode_case(CONFIGS["tiny"], device="cuda")
    assert_close(run(case), oracle(case), what="tiny")


def test_llama3_8b_config_full():
    case = make_decode_case(CONFIGS["llama3_8b_b64"], device="cuda")
    assert_close(run(case), oracle(case), what="llama3_8b_b64")


EDGE = [1, 2, 15, 16, 17, 31, 32, 33, 48, 100, 513, 1000]


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("B", [16, 32])
@pytest.mark.parametrize("g", [1, 2, 4, 8, 16])
def test_shapes_and_edge_lengths(dtype, d, B, g):
    Hkv = 2
    cfg = small_cfg(EDGE, Hq=Hkv * g, Hkv=Hkv, d=d, B=B, dtype=dtype, seed=11 + g + d + B)
    case = make_decode_case(cfg, device="cuda")
    assert_close(run(case), oracle(case), what=f"{dtype} d{d} B{B} g{g}")


def test_poisoned_memory_is_never_read():
    cfg = small_cfg([1, 15, 17, 40, 63, 300], Hq=16, Hkv=2)
    clean = make_decode_case(cfg, device="cuda")
    dirty = make_decode_case(cfg, device="cuda", poison_unused=True)
    # same values where it matters: poisoning only touched unused slots/entries
    a, b = run(clean), run(dirty)
    assert torch.isfinite(b.float()).all()
    assert torch.equal(a, b)
    assert_close(b, oracle(clean), what="poisoned")


def test_bitwise_invariant_to_block_placement():
    cfg = small_cfg([5, 16, 77, 301, 1200, 2049], Hq=32, Hkv=4)
    case = make_decode_case(cfg, device="cuda")
    base = run(case)
    g = torch.Generator(device="cpu").manual_seed(3)
    for _ in range(3):
        relabel = torch.randperm(case.num_blocks, generator=g)
        k2 = torch.empty_like(case.k_pool)
        v2 = torch.empty_like(case.v_pool)
        k2[relabel.cuda()] = case.k_pool
        v2[relabel.cuda()] = case.v_pool
        t2 = case.block_tables.copy()
        m = t2 >= 0
        t2[m] = relabel.numpy()[t2[m]]
        bt = torch.from_numpy(t2).cuda()
        cl = torch.from_numpy(case.context_lens).cuda()
        out = pa().pa_decode(case.q, k2, v2, bt, cl, case.scale)
        assert torch.equal(out, base)


def test_single_token_returns_value_exactly():
    cfg = small_cfg([1, 1, 1], Hq=8, Hkv=2, dtype="bf16")
    case = make_decode_case(cfg, device="cuda")
    out = run(case)
    for s in range(3):
        blk = int(case.block_tables[s, 0])
        for h in range(8):
            assert torch.equal(out[s, h], case.v_pool[blk, h // 4, 0])


def test_empty_and_mixed_contexts():
    cfg = small_cfg([0, 33, 0, 1, 0], Hq=8, Hkv=2)
    case = make_decode_case(cfg, device="cuda")
    out = torch.full_like(case.q, float("nan"))
    run(case, out=out)
    ref = oracle(case)
    assert torch.equal(out[0], torch.zeros_like(out[0]))
    assert torch.equal(out[2], torch.zeros_like(out[2]))
    assert_close(out, ref, what="mixed")


def test_all_contexts_empty():
    cfg = small_cfg([0, 0], Hq=4, Hkv=4, d=64)
    case = make_decode_case(cfg, device="cuda")
    out = torch.full_like(case.q, 7.0)
    run(case, out=out)
    assert torch.equal(out, torch.zeros_like(out))


def test_deterministic():
    cfg = small_cfg([3000, 17, 5000, 4096, 1, 777] * 4, Hq=64, Hkv=8)
    case = make_decode_case(cfg, device="cuda")
    bt, cl = dev_case(case)
    ws = pa().workspace_for(case.q, case.k_pool, bt)
    a = pa().pa_decode(case.q, case.k_pool, case.v_pool, bt, cl, case.scale, workspace=ws)
    b = pa().pa_decode(case.q, case.k_pool, case.v_pool, bt, cl, case.scale, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    assert_close(a, oracle(case), what="long/short mix")


def test_dirty_workspace_shared_across_shapes():
    """One scratch buffer, pre-filled with junk, serves calls of different
    batch sizes in both orders: the counters are cleared by every call."""
    small = make_decode_case(small_cfg([700, 1300, 90], Hq=16, Hkv=2, seed=21), device="cuda")
    large = make_decode_case(small_cfg([2500, 40, 1900, 3333, 5, 1000] * 8, Hq=32, Hkv=8, seed=22), device="cuda")
    need = max(pa().pa_decode_workspace_bytes(c.q, c.k_pool, torch.from_numpy(c.block_tables))
               for c in (small, large))
    ws = torch.full((need,), 0xAB, dtype=torch.uint8, device="cuda")
    ref_s, ref_l = oracle(small), oracle(large)
    for order in ((small, large, small), (large, small, large)):
        for c in order:
            bt, cl = dev_case(c)
            out = pa().pa_decode(c.q, c.k_pool, c.v_pool, bt, cl, c.scale, workspace=ws)
            assert_close(out, ref_s if c is small else ref_l, what="shared workspace")


def test_error_word_stays_clear_on_good_input():
    case = make_decode_case(CONFIGS["tiny"], device="cuda")
    err = pa().new_error_word("cuda")
    run(case, err=err)
    assert pa().pa_read_error(err) == 0


def sample_rows(case, n, seed):
    r = np.random.Generator(np.random.PCG64(seed))
    N, Hq = case.q.shape[0], case.q.shape[1]
    ctx = case.context_lens
    pick = {int(np.argmax(ctx)), int(np.argmin(ctx))} | set(int(x) for x in r.integers(0, N, size=n))
    rows = sorted({(s, int(h)) for s in pick for h in r.integers(0, Hq, size=2)})
    return rows


def test_llama3_70b_batch256_full_size_sampled():
    """The headline workload at full size, in the bench's launch configuration."""
    case = make_decode_case(CONFIGS["llama3_70b_b256"], device="cuda")
    out = run(case)
    assert torch.isfinite(out.float()).all()
    rows = sample_rows(case, 12, 5)
    assert_close(out, oracle(case, rows=rows), rows=rows, what="llama3_70b_b256")


def test_long_context_mha_full_size_sampled():
    case = make_decode_case(CONFIGS["long_mha_32k"], device="cuda")
    out = run(case)
    assert torch.isfinite(out.float()).all()
    rows = sample_rows(case, 2, 6)[:4]
    assert_close(out, oracle(case, rows=rows), rows=rows, what="long_mha_32k")
    del case
    torch.cuda.empty_cache()


# ---- peaked softmaxes: the running maximum moves, one weight dominates ----
PEAK = [(8.0, 0.0), (32.0, 0.0), (2.0, 6.0)]      # (q multiplier, K growth along the context)
MIX = (3000, 17, 5000, 4096, 1, 777, 33, 1500)    # pairs cut by chunk boundaries, and short ones


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("d,B,g,Hkv", [(128, 16, 8, 8), (128, 32, 16, 4), (64, 16, 1, 8), (128, 16, 4, 4)])
@pytest.mark.parametrize("q_mult,k_growth", PEAK)
def test_peaked_softmax(dtype, d, B, g, Hkv, q_mult, k_growth):
    cfg = small_cfg(MIX, Hq=Hkv * g, Hkv=Hkv, d=d, B=B, dtype=dtype, seed=200 + d + B + g)
    case = make_decode_case(cfg, device="cuda")
    sharpen(case, q_mult, k_growth)
    assert_close(run(case), oracle(case), what=f"peaked {dtype} d{d} B{B} g{g} x{q_mult} +{k_growth}")


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_dominant_key_late_in_a_split_context(dtype):
    # one key per sequence far above the rest, planted in the last blocks of
    # long contexts (after many stages and chunk boundaries) or at the start
    cfg = small_cfg(MIX, Hq=64, Hkv=8, dtype=dtype, seed=241)
    case = make_decode_case(cfg, device="cuda")
    for s, n in enumerate(case.context_lens):
        plant_key(case, s, int(n) - 1 - (s % 3) * 7 if n > 21 else 0)
    assert_close(run(case), oracle(case), what=f"dominant late key {dtype}")


def test_32k_contexts_with_the_maximum_in_a_middle_piece():
    # multi-head 32K contexts are cut into many pieces; the dominant key sits
    # in a middle piece, so the merge's exp(m_p - M) factors decide the result
    cfg = small_cfg([32768, 32768], Hq=8, Hkv=8, dtype="bf16", seed=251)
    case = make_decode_case(cfg, device="cuda")
    sharpen(case, 2.0)
    plant_key(case, 0, 16000, target=12.0)
    plant_key(case, 1, 20001, target=25.0)
    assert_close(run(case), oracle(case), what="32K, maximum in a middle piece")


def test_llama3_70b_batch256_peaked_sampled():
    case = make_decode_case(CONFIGS["llama3_70b_b256"], device="cuda", seed=1013)
    sharpen(case, 8.0)
    out = run(case)
    rows = sample_rows(case, 10, 15)
    assert_close(out, oracle(case, rows=rows), rows=rows, what="llama3_70b_b256 peaked")
