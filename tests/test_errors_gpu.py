"""Bad data found on the device sets the error word and poisons only the
affected rows; nothing traps.  All faults are injected from the host side
(bad table entries / lengths that the kernel's own checks catch)."""

import numpy as np
import pytest
import torch

from oracle.attention import decode_ref
from tests.gpu_util import assert_close, need_gpu
from workloads import DecodeConfig, make_decode_case

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()


def pa():
    import paged_kv_cache_254_gb300 as m
    return m


def case_with(ctx, Hq=16, Hkv=2):
    cfg = DecodeConfig(name="err", num_seqs=len(ctx), num_q_heads=Hq, num_kv_heads=Hkv, head_dim=128,
                       block_size=16, dtype="bf16", seed=31, ctx_fixed=tuple(ctx), pool_factor=1.5)
    return make_decode_case(cfg, device="cuda")


def decode(case, tables, ctx):
    err = pa().new_error_word("cuda")
    out = pa().pa_decode(case.q, case.k_pool, case.v_pool, torch.from_numpy(tables).cuda(),
                         torch.from_numpy(ctx).cuda(), case.scale, err=err)
    return out, err


def test_bad_block_id_poisons_its_sequence_only():
    case = case_with([300, 200, 40, 1000])
    good_ref = decode_ref(case.q, case.k_pool, case.v_pool, case.block_tables, case.context_lens, case.scale)
    tables = case.block_tables.copy()
    tables[1, 5] = case.num_blocks + 3          # inside the context of sequence 1
    out, err = decode(case, tables, case.context_lens.copy())
    assert pa().pa_read_error(err) == 4
    assert int(err.item()) == 1
    assert torch.isnan(out[1].float()).all()
    keep = [0, 2, 3]
    assert_close(out[keep], good_ref[keep], what="rows without the bad block")


def test_negative_block_id_is_caught():
    case = case_with([64, 65])
    tables = case.block_tables.copy()
    tables[0, 0] = -5
    out, err = decode(case, tables, case.context_lens.copy())
    assert int(err.item()) == 1
    assert torch.isnan(out[0].float()).all()
    assert torch.isfinite(out[1].float()).all()


def test_bad_context_length_poisons_its_rows():
    case = case_with([100, 50, 70])
    ctx = case.context_lens.copy()
    mb = case.block_tables.shape[1]
    ctx[0] = mb * 16 + 1                        # longer than the table can hold
    ctx[2] = -4
    out, err = decode(case, case.block_tables, ctx)
    assert pa().pa_read_error(err) == 4
    assert int(err.item()) == 2
    assert torch.isnan(out[0].float()).all() and torch.isnan(out[2].float()).all()
    ref = decode_ref(case.q, case.k_pool, case.v_pool, case.block_tables, case.context_lens, case.scale,
                     rows=[(1, h) for h in range(16)])
    assert_close(out, ref, rows=[(1, h) for h in range(16)], what="good row")


def test_unsupported_shapes_raise():
    case = case_with([10])
    q3 = torch.zeros((1, 6, 128), dtype=torch.bfloat16, device="cuda")   # 6 / 2 = group of 3
    with pytest.raises(pa().PagedAttentionError, match="UNSUPPORTED"):
        pa().pa_decode(q3, case.k_pool, case.v_pool, torch.from_numpy(case.block_tables).cuda(),
                       torch.from_numpy(case.context_lens).cuda(), case.scale)
    with pytest.raises(ValueError):
        pa().pa_decode(case.q.cpu(), case.k_pool, case.v_pool, torch.from_numpy(case.block_tables).cuda(),
                       torch.from_numpy(case.context_lens).cuda(), case.scale)
    small_ws = torch.zeros(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(pa().PagedAttentionError, match="WORKSPACE"):
        pa().pa_decode(case.q, case.k_pool, case.v_pool, torch.from_numpy(case.block_tables).cuda(),
                       torch.from_numpy(case.context_lens).cuda(), case.scale, workspace=small_ws)


def test_a_wait_that_runs_out_sets_timeout_and_the_call_returns():
    """Fault injection on the host side: every worker's first stage wait is
    made on a barrier that nothing completes, with a 200 us limit.  The kernel
    must report PA_ERR_TIMEOUT, write NaN to every row (also the rows of pairs
    split across chunks, which go through the merge), drain its copies and
    return; the next call at the normal limit is clean and correct."""
    from oracle.attention import decode_ref
    case = case_with([3000, 17, 5000, 4096, 1, 777] * 4, Hq=64, Hkv=8)
    want = decode_ref(case.q, case.k_pool, case.v_pool, case.block_tables, case.context_lens, case.scale)
    pa().pa_set_decode_stall_ns(200_000)
    try:
        out, err = decode(case, case.block_tables, case.context_lens.copy())
        assert pa().pa_read_error(err) == 5                  # PA_ERR_TIMEOUT
        assert int(err.item()) & 16
        assert torch.isnan(out.float()).all()
    finally:
        pa().pa_set_decode_stall_ns(0)
    out, err = decode(case, case.block_tables, case.context_lens.copy())
    assert pa().pa_read_error(err) == 0
    assert_close(out, want, what="after the timeout")


@pytest.mark.parametrize("kind", ["fp8", "int4"])
def test_timeout_path_of_the_quantized_decodes(kind):
    from workloads import make_codes, make_int4_pool
    case = case_with([700, 2000, 33], Hq=16, Hkv=2)
    g = torch.Generator(device="cuda").manual_seed(77)
    bt = torch.from_numpy(case.block_tables).cuda()
    cl = torch.from_numpy(case.context_lens).cuda()
    if kind == "fp8":
        pool = make_codes((case.num_blocks, 2, 2, 16, 128), g, "cuda")
        run = lambda err: pa().pa_decode_fp8(case.q, pool, bt, cl, case.scale, 0.25, 0.25, err=err)  # noqa: E731
    else:
        pool = make_int4_pool(case.num_blocks, 2, 16, 128, g, "cuda")
        run = lambda err: pa().pa_decode_int4(case.q, pool, bt, cl, case.scale, err=err)  # noqa: E731
    pa().pa_set_decode_stall_ns(100_000)
    try:
        err = pa().new_error_word("cuda")
        out = run(err)
        assert pa().pa_read_error(err) == 5
        assert torch.isnan(out.float()).all()
    finally:
        pa().pa_set_decode_stall_ns(0)
    err = pa().new_error_word("cuda")
    out = run(err)
    assert pa().pa_read_error(err) == 0
    assert torch.isfinite(out.float()).all()
