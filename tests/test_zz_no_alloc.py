"""The decode entry point that allocates nothing (pa_decode_noalloc).

It serves callers that cannot allocate device memory -- a framework that has
already reserved the device's memory for its own pool, a plugin host that
passes only inputs and outputs, a serving loop that cannot afford the device
synchronisation cudaMalloc/cudaFree may cause.  Its scratch is a fixed static
buffer inside libpa.so.  This file is collected last so that a stop-at-first-
failure run has already run every other test.
"""

import ctypes

import numpy as np
import pytest
import torch

from paged_kv_cache_254_gb300 import _lib
from tests.gpu_util import ATOL, RTOL, assert_close, dev_case, need_gpu
from workloads import DecodeConfig, make_decode_case

pytestmark = pytest.mark.gpu


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def test_noalloc_matches_oracle_and_pa_decode_on_two_calls_in_a_row():
    need_gpu()
    import paged_kv_cache_254_gb300 as pa
    from oracle.attention import decode_ref

    # lengths that split sequences across chunks, so the scratch is really used
    cfg = DecodeConfig(name="noalloc", num_seqs=24, num_q_heads=64, num_kv_heads=8, head_dim=128,
                       block_size=16, dtype="bf16", seed=41, ctx_fixed=(3000, 17, 5000, 4096, 1, 777) * 4,
                       pool_factor=1.2)
    case = make_decode_case(cfg, device="cuda")
    bt, cl = dev_case(case)
    ref = decode_ref(case.q, case.k_pool, case.v_pool, case.block_tables, case.context_lens, case.scale)
    want = pa.pa_decode(case.q, case.k_pool, case.v_pool, bt, cl, case.scale).double()

    lib = _lib.load()
    shape = pa.make_shape(cfg.num_seqs, cfg.num_q_heads, cfg.num_kv_heads, cfg.head_dim, cfg.block_size,
                          case.num_blocks, cfg.max_blocks_per_seq, case.q.dtype)
    err = pa.new_error_word("cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for _ in range(2):
        out = torch.full_like(case.q, float("nan"))
        st = lib.pa_decode_noalloc(ctypes.byref(shape), _ptr(case.q), _ptr(case.k_pool), _ptr(case.v_pool),
                                   _ptr(bt), _ptr(cl), ctypes.c_float(case.scale), _ptr(out), _ptr(err), stream)
        assert st == 0, _lib.status_string(st)
        torch.cuda.synchronize()
        got = out.double()
        assert torch.isfinite(got).all()
        # the same tolerance as every decode parity test, against the fp64
        # oracle and against pa_decode with a caller-owned workspace
        assert_close(out, ref, what="no-alloc decode vs oracle")
        assert ((got - want).abs() <= ATOL + RTOL * want.abs()).all()
    assert lib.pa_read_error(_ptr(err), stream) == 0


def test_noalloc_rejects_shapes_beyond_its_buffer():
    need_gpu()
    import paged_kv_cache_254_gb300 as pa

    lib = _lib.load()
    # 5M sequences need 40 MB of per-sequence prefix sums alone, past the
    # 32 MiB static buffer even at the minimum scratch.  The size check comes
    # before every other check, so the call refuses with null pointers (and
    # were it ever to pass, pa_decode's null check would still refuse).
    shape = pa.make_shape(5_000_000, 64, 8, 128, 16, 1000, 8, torch.bfloat16)
    null = ctypes.c_void_p(0)
    assert (5_000_000 + 1) * 8 > _lib.NOALLOC_SCRATCH_BYTES
    assert lib.pa_decode_workspace_bytes(ctypes.byref(shape)) > _lib.NOALLOC_SCRATCH_BYTES
    st = lib.pa_decode_noalloc(ctypes.byref(shape), null, null, null, null, null, ctypes.c_float(0.1), null,
                               null, null)
    assert st == 6   # PA_ERR_WORKSPACE
