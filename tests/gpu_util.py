"""Shared helpers of the GPU parity tests."""

import numpy as np
import pytest
import torch

# Attention tolerance: |gpu - oracle| <= ATOL + RTOL * |oracle| per element
# (max abs 2e-3 and max rel 1e-2 combined in allclose form, because a
# bf16 output rounding alone can exceed 2e-3 for |x| >= 1).
ATOL, RTOL = 2e-3, 1e-2


def need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from paged_kv_cache_254_gb300 import _build
    _build.build()


def dev_case(case, device="cuda"):
    """Block tables and context lengths of a workload as device int32."""
    bt = torch.from_numpy(np.ascontiguousarray(case.block_tables)).to(device)
    cl = torch.from_numpy(np.ascontiguousarray(case.context_lens)).to(device)
    return bt, cl


def assert_close(got, ref, rows=None, what=""):
    """got: GPU tensor [N, Hq, d]; ref: fp64 array of the same shape (NaN rows
    are skipped when ``rows`` is given)."""
    g = got.detach().double().cpu().numpy()
    if rows is not None:
        idx = tuple(np.array(rows).T)
        g, ref = g[idx], ref[idx]
    assert np.isfinite(ref).all()
    assert np.isfinite(g).all(), f"{what}: non-finite GPU output"
    err = np.abs(g - ref)
    bound = ATOL + RTOL * np.abs(ref)
    worst = np.argmax(err - bound)
    assert (err <= bound).all(), (f"{what}: max abs err {err.max():.3e}, worst element err "
                                  f"{err.flat[worst]:.3e} vs bound {bound.flat[worst]:.3e} "
                                  f"(ref {ref.flat[worst]:.4f}, got {g.flat[worst]:.4f})")
    return float(err.max())


def from_bits(arr, dtype):
    """Host tensor of `dtype` (fp16 / bf16) viewing an int16 bit-pattern array."""
    return torch.from_numpy(np.ascontiguousarray(arr)).view(dtype)
