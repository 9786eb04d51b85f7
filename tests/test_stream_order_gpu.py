"""Calls queued back to back on one stream, sharing one workspace, with no host
synchronisation in between.

Within a call the attention kernel starts while the pre-pass runs and the merge
while the attention kernel retires (programmatic dependent launch); across
calls each pre-pass clears the counters the previous call's kernels used.  The
outputs of every call are kept and compared with the fp64 oracle only after the
whole queue has run, so a merge reading a later call's partial states, or a
kernel reading counters before they are cleared, shows up as a wrong row."""

import numpy as np
import pytest
import torch

from oracle.attention import decode_multi_ref, decode_ref
from tests.gpu_util import assert_close, dev_case, need_gpu
from workloads import DecodeConfig, make_decode_case, make_values

pytestmark = pytest.mark.gpu

WS_BYTES = 64 << 20


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()


def pa():
    import paged_kv_cache_254_gb300 as m
    return m


def decode_case(ctx, Hq, Hkv, B=16, seed=7):
    cfg = DecodeConfig(name="queued", num_seqs=len(ctx), num_q_heads=Hq, num_kv_heads=Hkv, head_dim=128,
                       block_size=B, dtype="bf16", seed=seed, ctx_fixed=tuple(ctx), pool_factor=1.5)
    return make_decode_case(cfg, device="cuda")


def multi_inputs(case, qlens, seed):
    qs = np.concatenate([[0], np.cumsum(qlens)]).astype(np.int32)
    gen = torch.Generator(device="cuda").manual_seed(seed)
    q = make_values((int(qs[-1]), case.q.shape[1], case.q.shape[2]), "bf16", gen, "cuda")
    return q, qs


def queue_decode(case, ws):
    bt, cl = dev_case(case)
    return pa().pa_decode(case.q, case.k_pool, case.v_pool, bt, cl, case.scale, workspace=ws)


def queue_multi(case, q, qs, max_q, ws):
    bt, cl = dev_case(case)
    return pa().pa_decode_multi(q, case.k_pool, case.v_pool, bt, cl, torch.from_numpy(qs).cuda(), case.scale,
                                max_q_len=max_q, workspace=ws)


def test_decode_calls_queued_on_one_workspace():
    # two batches whose long pairs are cut into several pieces, alternated
    a = decode_case([9000, 17, 5000, 4096, 1, 777, 12000, 300], Hq=32, Hkv=4, seed=41)
    b = decode_case([33, 7000, 15000, 2, 2500, 640], Hq=16, Hkv=2, B=32, seed=42)
    ws = torch.full((WS_BYTES,), 0xCD, dtype=torch.uint8, device="cuda")
    order = (a, b, a, b, a)
    outs = [queue_decode(c, ws) for c in order]
    torch.cuda.synchronize()
    refs = {id(a): decode_ref(a.q, a.k_pool, a.v_pool, a.block_tables, a.context_lens, a.scale),
            id(b): decode_ref(b.q, b.k_pool, b.v_pool, b.block_tables, b.context_lens, b.scale)}
    for i, (c, out) in enumerate(zip(order, outs)):
        assert_close(out, refs[id(c)], what=f"queued decode call {i}")
    assert torch.equal(outs[0], outs[2]) and torch.equal(outs[0], outs[4])
    assert torch.equal(outs[1], outs[3])


def test_decode_and_multi_token_calls_queued_on_one_workspace():
    # a decode, a 2-token (mma.sync) and a 4-token (tcgen05) launch over the
    # same pools, interleaved on one stream and one workspace
    case = decode_case([8000, 50, 3000, 11000, 129, 6000], Hq=16, Hkv=2, seed=43)
    q2, qs2 = multi_inputs(case, [2, 1, 2, 2, 2, 0], seed=44)       # up to 16 rows per pair: mma.sync
    q4, qs4 = multi_inputs(case, [4, 3, 4, 1, 4, 4], seed=45)       # up to 32 rows per pair: tcgen05
    ws = torch.full((WS_BYTES,), 0x5A, dtype=torch.uint8, device="cuda")
    outs = []
    for _ in range(2):
        outs.append(("decode", queue_decode(case, ws)))
        outs.append(("q2", queue_multi(case, q2, qs2, 2, ws)))
        outs.append(("q4", queue_multi(case, q4, qs4, 4, ws)))
    torch.cuda.synchronize()
    refs = {"decode": decode_ref(case.q, case.k_pool, case.v_pool, case.block_tables, case.context_lens,
                                 case.scale),
            "q2": decode_multi_ref(q2, case.k_pool, case.v_pool, case.block_tables, case.context_lens, qs2,
                                   case.scale),
            "q4": decode_multi_ref(q4, case.k_pool, case.v_pool, case.block_tables, case.context_lens, qs4,
                                   case.scale)}
    for i, (kind, out) in enumerate(outs):
        assert_close(out, refs[kind], what=f"queued call {i} ({kind})")
    for k in range(3):
        assert torch.equal(outs[k][1], outs[k + 3][1]), outs[k][0]
