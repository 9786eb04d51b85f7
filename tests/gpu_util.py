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


def sharpen(case, q_mult=1.0, k_growth=0.0):
    """Make the decode softmaxes peaked instead of nearly flat.

    q is multiplied by ``q_mult``, which widens the spread of the scores by the
    same factor.  With ``k_growth`` every sequence's K row at context position t
    is multiplied by 1 + k_growth * (t + 1) / ctx, so later keys score higher and
    the running maximum keeps rising along the context -- across blocks,
    stages, chunks and split pieces.  The tensors are changed in place and
    re-rounded to their dtype; the oracle reads the same tensors."""
    if q_mult != 1.0:
        case.q.mul_(q_mult)
    if k_growth:
        B = case.k_pool.shape[2]
        dev = case.k_pool.device
        for s, n in enumerate(case.context_lens):
            n = int(n)
            nb = -(-n // B)
            if nb == 0:
                continue
            ids = torch.from_numpy(case.block_tables[s, :nb].astype(np.int64)).to(dev)
            t = torch.arange(nb * B, device=dev, dtype=torch.float32).reshape(nb, B)
            f = 1.0 + k_growth * (t + 1.0) / n
            case.k_pool[ids] = (case.k_pool[ids].float() * f[:, None, :, None]).to(case.k_pool.dtype)


def plant_key(case, s, t, target=30.0, q=None):
    """Make cached token t of sequence s dominate: for every KV head its K row
    becomes q[s, first head of the group] scaled so that this head's score is
    `target` (natural-log units), far above the others.  ``q`` defaults to
    case.q [N, Hq, d] (a multi-token test passes the row it wants)."""
    q = case.q if q is None else q
    Hq, Hkv, B = q.shape[-2], case.k_pool.shape[1], case.k_pool.shape[2]
    g = Hq // Hkv
    blk, off = int(case.block_tables[s, t // B]), t % B
    for kh in range(Hkv):
        qv = (q[s, kh * g] if q.dim() == 3 else q[kh * g]).float()
        k = qv * (target / (case.scale * float(qv @ qv)))
        case.k_pool[blk, kh, off] = k.to(case.k_pool.dtype)
