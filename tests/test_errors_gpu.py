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
