"""KV append and copy-on-write block copy: bit-exact against the oracle,
including untouched slots; bad slots / pairs set the error word."""

import numpy as np
import pytest
import torch

from oracle.attention import decode_ref
from oracle.kv_ops import append_ref, bits, copy_ref, slot_of
from tests.gpu_util import assert_close, dev_case, from_bits, need_gpu
from workloads import CONFIGS, SAMPLING, make_decode_case, make_sampling_case, make_values, sampling_tables

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()


def pa():
    import paged_kv_cache_254_gb300 as m
    return m


def pools(NB, Hkv, B, d, dtype, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    return make_values((NB, Hkv, B, d), dtype, g, "cuda"), make_values((NB, Hkv, B, d), dtype, g, "cuda")


@pytest.mark.parametrize("dtype,d,B", [("bf16", 128, 16), ("fp16", 64, 32), ("bf16", 64, 16)])
def test_append_bit_exact(dtype, d, B):
    NB, Hkv, T = 50, 4, 300
    kp, vp = pools(NB, Hkv, B, d, dtype, 1)
    g = torch.Generator(device="cuda").manual_seed(2)
    kn = make_values((T, Hkv, d), dtype, g, "cuda")
    vn = make_values((T, Hkv, d), dtype, g, "cuda")
    r = np.random.Generator(np.random.PCG64(3))
    slots = r.permutation(NB * B)[:T].astype(np.int64)
    slots[::7] = -1                                   # padding rows
    want_k, want_v = append_ref(bits(kp), bits(vp), bits(kn), bits(vn), slots, B)
    pa().pa_append_kv(kn, vn, torch.from_numpy(slots).cuda(), kp, vp)
    torch.cuda.synchronize()
    assert np.array_equal(bits(kp), want_k)
    assert np.array_equal(bits(vp), want_v)


def test_append_rejects_slot_past_pool():
    NB, Hkv, B, d = 8, 2, 16, 64
    kp, vp = pools(NB, Hkv, B, d, "bf16", 4)
    before = bits(kp)
    kn = torch.ones((2, Hkv, d), dtype=torch.bfloat16, device="cuda")
    err = pa().new_error_word("cuda")
    pa().pa_append_kv(kn, kn, torch.tensor([NB * B, 10 ** 9], dtype=torch.int64, device="cuda"), kp, vp, err=err)
    assert pa().pa_read_error(err) == 4                 # PA_ERR_OUT_OF_RANGE
    assert int(err.item()) == 4                          # the slot bit
    assert np.array_equal(bits(kp), before)


@pytest.mark.parametrize("dtype,d,B,Hkv", [("bf16", 128, 32, 8), ("fp16", 64, 16, 2)])
def test_copy_blocks_bit_exact(dtype, d, B, Hkv):
    NB = 40
    kp, vp = pools(NB, Hkv, B, d, dtype, 5)
    pairs = np.array([[3, 10], [3, 11], [7, 12], [0, 39], [5, 5]], dtype=np.int32)
    want_k, want_v = copy_ref(bits(kp), bits(vp), pairs)
    pa().pa_copy_blocks(torch.from_numpy(pairs).cuda(), kp, vp)
    torch.cuda.synchronize()
    assert np.array_equal(bits(kp), want_k)
    assert np.array_equal(bits(vp), want_v)


def test_copy_many_pairs_grid_stride():
    NB, Hkv, B, d = 1200, 1, 16, 64
    kp, vp = pools(NB, Hkv, B, d, "bf16", 6)
    r = np.random.Generator(np.random.PCG64(7))
    perm = r.permutation(NB)
    pairs = np.stack([perm[:600], perm[600:]], axis=1).astype(np.int32)
    want_k, want_v = copy_ref(bits(kp), bits(vp), pairs)
    pa().pa_copy_blocks(torch.from_numpy(pairs).cuda(), kp, vp)
    torch.cuda.synchronize()
    assert np.array_equal(bits(kp), want_k)
    assert np.array_equal(bits(vp), want_v)


def test_copy_rejects_bad_pair():
    kp, vp = pools(6, 2, 16, 64, "fp16", 8)
    before = bits(kp)
    err = pa().new_error_word("cuda")
    pa().pa_copy_blocks(torch.tensor([[1, 6], [-1, 2]], dtype=torch.int32, device="cuda"), kp, vp, err=err)
    assert pa().pa_read_error(err) == 4
    assert int(err.item()) == 8
    assert np.array_equal(bits(kp), before)


def test_decode_step_with_append():
    """Llama-3-8B-shaped step: append each sequence's newest token at position
    ctx-1, then decode over the updated cache."""
    case = make_decode_case(CONFIGS["llama3_8b_b64"], device="cuda")
    B = case.cfg.block_size
    slots = np.array([slot_of(case.block_tables[s], int(case.context_lens[s]) - 1, B)
                      for s in range(len(case.context_lens))], dtype=np.int64)
    want_k, want_v = append_ref(bits(case.k_pool), bits(case.v_pool), bits(case.k_new), bits(case.v_new), slots, B)
    pa().pa_append_kv(case.k_new, case.v_new, torch.from_numpy(slots).cuda(), case.k_pool, case.v_pool)
    bt, cl = dev_case(case)
    out = pa().pa_decode(case.q, case.k_pool, case.v_pool, bt, cl, case.scale)
    torch.cuda.synchronize()
    assert np.array_equal(bits(case.k_pool), want_k)
    assert np.array_equal(bits(case.v_pool), want_v)
    dt = case.q.dtype
    ref = decode_ref(case.q, from_bits(want_k, dt), from_bits(want_v, dt), case.block_tables, case.context_lens,
                     case.scale)
    assert_close(out, ref, what="append + decode")


@pytest.mark.parametrize("groups", [3, None])
def test_parallel_sampling_copy_append_decode(groups):
    """Shared prompt, copy-on-write of the half-full last prompt block, append
    of each sample's divergent tail plus its new token, then decode."""
    case = make_sampling_case(SAMPLING, device="cuda", groups=groups)
    cfg = case.cfg
    B = cfg.block_size
    tables, ctx = sampling_tables(case)
    S = cfg.samples
    pairs = np.array([[case.prompt_blocks[i // S][-1], case.private_last[i]]
                      for i in range(len(ctx)) if case.private_last[i] >= 0], dtype=np.int32)
    slots = np.concatenate([[slot_of(tables[i], t, B) for t in range(cfg.prompt_len, int(ctx[i]))]
                            for i in range(len(ctx))]).astype(np.int64)
    assert slots.size == case.k_new.shape[0]
    k0, v0 = bits(case.k_pool), bits(case.v_pool)
    wk, wv = copy_ref(k0, v0, pairs)
    wk, wv = append_ref(wk, wv, bits(case.k_new), bits(case.v_new), slots, B)

    pa().pa_copy_blocks(torch.from_numpy(pairs).cuda(), case.k_pool, case.v_pool)
    pa().pa_append_kv(case.k_new, case.v_new, torch.from_numpy(slots).cuda(), case.k_pool, case.v_pool)
    bt = torch.from_numpy(tables).cuda()
    cl = torch.from_numpy(ctx).cuda()
    out = pa().pa_decode(case.q, case.k_pool, case.v_pool, bt, cl, case.scale)
    torch.cuda.synchronize()
    assert np.array_equal(bits(case.k_pool), wk)
    assert np.array_equal(bits(case.v_pool), wv)
    r = np.random.Generator(np.random.PCG64(9))
    rows = sorted({(int(s), int(h)) for s in r.integers(0, len(ctx), size=10) for h in r.integers(0, 32, size=2)})
    if groups is not None:
        rows = None
    dt = case.q.dtype
    ref = decode_ref(case.q, from_bits(wk, dt), from_bits(wv, dt), tables, ctx, case.scale, rows=rows)
    assert_close(out, ref, rows=rows, what=f"sampling groups={groups}")
