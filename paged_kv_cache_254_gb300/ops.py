"""Python entry points with the C ABI's names: torch tensors in, kernels run.

PyTorch supplies device memory and streams only.  Each function checks that
its tensors sit on one CUDA device with the expected dtype and layout, then
calls the matching ``pa_*`` function of libpa.so on the current stream.
"""

from __future__ import annotations

import ctypes
import threading

import torch

from . import _lib

_DTYPES = {torch.float16: _lib.PA_FP16, torch.bfloat16: _lib.PA_BF16}


def _ptr(t) -> ctypes.c_void_p:
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _stream(device, stream=None) -> ctypes.c_void_p:
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return ctypes.c_void_p(s.cuda_stream)


def _need_cuda(name, t, dtype=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (there is no CPU path)")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")


def make_shape(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, max_blocks_per_seq,
               dtype) -> _lib.PaShape:
    return _lib.PaShape(int(num_seqs), int(num_q_heads), int(num_kv_heads), int(head_dim), int(block_size),
                        int(num_blocks), int(max_blocks_per_seq), _DTYPES[dtype])


def _pool_shape(k_pool, num_seqs=0, num_q_heads=1, max_blocks=1) -> _lib.PaShape:
    NB, Hkv, B, d = k_pool.shape
    return make_shape(num_seqs, num_q_heads, Hkv, d, B, NB, max_blocks, k_pool.dtype)


def pa_decode_workspace_bytes(q, k_pool, block_tables) -> int:
    N, Hq, _ = q.shape
    shape = _pool_shape(k_pool, N, Hq, block_tables.shape[1])
    with torch.cuda.device(q.device):
        return int(_lib.load().pa_decode_workspace_bytes(ctypes.byref(shape)))


_ws_lock = threading.Lock()
_ws_cache = {}


def workspace_for(q, k_pool, block_tables, stream=None) -> torch.Tensor:
    """A workspace kept per (device, stream) and grown on demand; pa_decode
    clears its counter region itself, so the buffer is reused as is."""
    need = pa_decode_workspace_bytes(q, k_pool, block_tables)
    if need == 0:
        return torch.empty(0, dtype=torch.uint8, device=q.device)
    s = stream if stream is not None else torch.cuda.current_stream(q.device)
    key = (q.device.index, s.cuda_stream)
    with _ws_lock:
        ws = _ws_cache.get(key)
        if ws is None or ws.numel() < need:
            ws = torch.zeros(max(need, 1 << 20), dtype=torch.uint8, device=q.device)
            _ws_cache[key] = ws
        return ws


def new_error_word(device) -> torch.Tensor:
    return torch.zeros(1, dtype=torch.int32, device=device)


def pa_decode(q, k_pool, v_pool, block_tables, context_lens, scale, out=None, workspace=None, err=None,
              stream=None):
    """out[N, Hq, d] = paged decode attention of q over the pools (see include/pa.h)."""
    _need_cuda("q", q)
    _need_cuda("k_pool", k_pool, q.dtype)
    _need_cuda("v_pool", v_pool, q.dtype)
    _need_cuda("block_tables", block_tables, torch.int32)
    _need_cuda("context_lens", context_lens, torch.int32)
    if q.dtype not in _DTYPES:
        raise TypeError("q must be float16 or bfloat16")
    if k_pool.shape != v_pool.shape or k_pool.dim() != 4 or q.dim() != 3:
        raise ValueError("q [N, Hq, d], k_pool and v_pool [NB, Hkv, B, d]")
    N, Hq, d = q.shape
    if k_pool.shape[3] != d or block_tables.dim() != 2 or block_tables.shape[0] != N or context_lens.shape != (N,):
        raise ValueError("shape mismatch between q, pools, block_tables and context_lens")
    if out is None:
        out = torch.empty_like(q)
    else:
        _need_cuda("out", out, q.dtype)
        if out.shape != q.shape:
            raise ValueError("out must have q's shape")
    if workspace is None:
        workspace = workspace_for(q, k_pool, block_tables, stream)
    else:
        _need_cuda("workspace", workspace)
    if err is not None:
        _need_cuda("err", err, torch.int32)
    shape = _pool_shape(k_pool, N, Hq, block_tables.shape[1])
    with torch.cuda.device(q.device):
        st = _lib.load().pa_decode(ctypes.byref(shape), _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(block_tables),
                                   _ptr(context_lens), ctypes.c_float(scale), _ptr(out), _ptr(workspace),
                                   ctypes.c_size_t(workspace.numel() * workspace.element_size()), _ptr(err),
                                   _stream(q.device, stream))
    _lib.check(st, "pa_decode")
    return out


def pa_append_kv(k_new, v_new, slot_mapping, k_pool, v_pool, err=None, stream=None):
    """Write k_new/v_new [T, Hkv, d] into the pools at slot_mapping [T] (int64; < 0 skips)."""
    _need_cuda("k_pool", k_pool)
    _need_cuda("v_pool", v_pool, k_pool.dtype)
    _need_cuda("k_new", k_new, k_pool.dtype)
    _need_cuda("v_new", v_new, k_pool.dtype)
    _need_cuda("slot_mapping", slot_mapping, torch.int64)
    T = slot_mapping.shape[0]
    if k_new.shape != (T,) + tuple(k_pool.shape[1:2]) + tuple(k_pool.shape[3:]) or v_new.shape != k_new.shape:
        raise ValueError("k_new, v_new must be [T, Hkv, d]")
    if err is not None:
        _need_cuda("err", err, torch.int32)
    shape = _pool_shape(k_pool)
    with torch.cuda.device(k_pool.device):
        st = _lib.load().pa_append_kv(ctypes.byref(shape), ctypes.c_int32(T), _ptr(k_new), _ptr(v_new),
                                      _ptr(slot_mapping), _ptr(k_pool), _ptr(v_pool), _ptr(err),
                                      _stream(k_pool.device, stream))
    _lib.check(st, "pa_append_kv")


def pa_copy_blocks(src_dst_pairs, k_pool, v_pool, err=None, stream=None):
    """Copy whole blocks src -> dst for each row of src_dst_pairs [n, 2] (int32)."""
    _need_cuda("k_pool", k_pool)
    _need_cuda("v_pool", v_pool, k_pool.dtype)
    _need_cuda("src_dst_pairs", src_dst_pairs, torch.int32)
    if src_dst_pairs.dim() != 2 or src_dst_pairs.shape[1] != 2:
        raise ValueError("src_dst_pairs must be [n, 2]")
    if err is not None:
        _need_cuda("err", err, torch.int32)
    shape = _pool_shape(k_pool)
    with torch.cuda.device(k_pool.device):
        st = _lib.load().pa_copy_blocks(ctypes.byref(shape), _ptr(src_dst_pairs),
                                        ctypes.c_int32(src_dst_pairs.shape[0]), _ptr(k_pool), _ptr(v_pool),
                                        _ptr(err), _stream(k_pool.device, stream))
    _lib.check(st, "pa_copy_blocks")


def pa_set_decode_stall_ns(wait_ns: int) -> None:
    """Fault injection for tests (see include/pa.h): with wait_ns > 0 every
    later decode launch makes each worker's first stage wait on a barrier
    that nothing completes, for at most wait_ns, so the kernel's timeout path
    runs; 0 turns it off."""
    _lib.check(_lib.load().pa_set_decode_stall_ns(ctypes.c_uint64(int(wait_ns))), "pa_set_decode_stall_ns")


def pa_read_error(err, stream=None) -> int:
    """Synchronise the stream and return the status the error word maps to."""
    _need_cuda("err", err, torch.int32)
    with torch.cuda.device(err.device):
        return int(_lib.load().pa_read_error(_ptr(err), _stream(err.device, stream)))


def pa_decode_shared_prefix(q, k_pool, v_pool, block_tables, context_lens, group_starts, group_prefix_blocks,
                            scale, out=None, workspace=None, err=None, stream=None):
    """Prefix-aware decode (see include/pa.h): group_starts [G + 1] and
    group_prefix_blocks [G] are int32 CUDA tensors describing sequences that
    share their leading blocks."""
    _need_cuda("q", q)
    _need_cuda("k_pool", k_pool, q.dtype)
    _need_cuda("v_pool", v_pool, q.dtype)
    _need_cuda("block_tables", block_tables, torch.int32)
    _need_cuda("context_lens", context_lens, torch.int32)
    _need_cuda("group_starts", group_starts, torch.int32)
    _need_cuda("group_prefix_blocks", group_prefix_blocks, torch.int32)
    n_groups = group_prefix_blocks.shape[0]
    if group_starts.shape != (n_groups + 1,):
        raise ValueError("group_starts must have one more entry than group_prefix_blocks")
    N, Hq, d = q.shape
    if k_pool.shape != v_pool.shape or k_pool.shape[3] != d or block_tables.shape[0] != N:
        raise ValueError("shape mismatch between q, pools and block_tables")
    if out is None:
        out = torch.empty_like(q)
    else:
        _need_cuda("out", out, q.dtype)
    shape = _pool_shape(k_pool, N, Hq, block_tables.shape[1])
    lib = _lib.load()
    with torch.cuda.device(q.device):
        need = int(lib.pa_decode_shared_prefix_workspace_bytes(ctypes.byref(shape)))
        if workspace is None:
            workspace = _shared_workspace(q.device, need, stream)
        else:
            _need_cuda("workspace", workspace)
        if err is not None:
            _need_cuda("err", err, torch.int32)
        st = lib.pa_decode_shared_prefix(ctypes.byref(shape), _ptr(q), _ptr(k_pool), _ptr(v_pool),
                                         _ptr(block_tables), _ptr(context_lens), ctypes.c_int32(n_groups),
                                         _ptr(group_starts), _ptr(group_prefix_blocks), ctypes.c_float(scale),
                                         _ptr(out), _ptr(workspace),
                                         ctypes.c_size_t(workspace.numel() * workspace.element_size()), _ptr(err),
                                         _stream(q.device, stream))
    _lib.check(st, "pa_decode_shared_prefix")
    return out


def pa_decode_multi(q, k_pool, v_pool, block_tables, context_lens, q_start, scale, max_q_len=None,
                    out=None, workspace=None, err=None, stream=None):
    """Multi-token query paged attention (see include/pa.h): q [T, Hq, d]
    holds each sequence's chunk of new tokens at rows q_start[b] ..
    q_start[b + 1] - 1 (q_start: int32 CUDA tensor [N + 1]); token i of a
    chunk attends causally to keys t <= ctx - q_len + i.  max_q_len defaults
    to the largest chunk (read from q_start on the host)."""
    _need_cuda("q", q)
    _need_cuda("k_pool", k_pool, q.dtype)
    _need_cuda("v_pool", v_pool, q.dtype)
    _need_cuda("block_tables", block_tables, torch.int32)
    _need_cuda("context_lens", context_lens, torch.int32)
    _need_cuda("q_start", q_start, torch.int32)
    T, Hq, d = q.shape
    N = block_tables.shape[0]
    if q_start.shape != (N + 1,) or context_lens.shape != (N,):
        raise ValueError("q_start must have N + 1 entries and context_lens N")
    if k_pool.shape != v_pool.shape or k_pool.shape[3] != d:
        raise ValueError("shape mismatch between q and the pools")
    if max_q_len is None:
        qs = q_start.cpu()
        max_q_len = max(1, int((qs[1:] - qs[:-1]).max().item())) if N > 0 else 1
    if out is None:
        out = torch.empty_like(q)
    else:
        _need_cuda("out", out, q.dtype)
        if out.shape != q.shape:
            raise ValueError("out must have q's shape")
    shape = _pool_shape(k_pool, N, Hq, block_tables.shape[1])
    lib = _lib.load()
    with torch.cuda.device(q.device):
        need = int(lib.pa_decode_multi_workspace_bytes(ctypes.byref(shape), ctypes.c_int32(max_q_len)))
        if need == 0 and workspace is None:
            # an invalid shape or chunk bound: let the call report which
            workspace = torch.empty(0, dtype=torch.uint8, device=q.device)
        elif workspace is None:
            workspace = _shared_workspace(q.device, need, stream)
        else:
            _need_cuda("workspace", workspace)
        if err is not None:
            _need_cuda("err", err, torch.int32)
        st = lib.pa_decode_multi(ctypes.byref(shape), ctypes.c_int32(max_q_len), ctypes.c_int32(T), _ptr(q),
                                 _ptr(q_start), _ptr(k_pool), _ptr(v_pool), _ptr(block_tables),
                                 _ptr(context_lens), ctypes.c_float(scale), _ptr(out), _ptr(workspace),
                                 ctypes.c_size_t(workspace.numel() * workspace.element_size()), _ptr(err),
                                 _stream(q.device, stream))
    _lib.check(st, "pa_decode_multi")
    return out


_sp_cache = {}


def _shared_workspace(device, need, stream=None):
    s = stream if stream is not None else torch.cuda.current_stream(device)
    key = (device.index, s.cuda_stream)
    with _ws_lock:
        ws = _sp_cache.get(key)
        if ws is None or ws.numel() < need:
            ws = torch.empty(max(need, 1 << 20), dtype=torch.uint8, device=device)
            _sp_cache[key] = ws
        return ws


KV_FORMATS = {"e4m3": _lib.PA_FP8_E4M3, "e5m2": _lib.PA_FP8_E5M2}


def _need_pool8(kv_pool):
    _need_cuda("kv_pool", kv_pool, torch.uint8)
    if kv_pool.dim() != 5 or kv_pool.shape[2] != 2:
        raise ValueError("kv_pool must be uint8 [NB, Hkv, 2, B, d] (the V half stored dims-first)")
    return kv_pool.shape[0], kv_pool.shape[1], kv_pool.shape[3], kv_pool.shape[4]


def pa_decode_fp8(q, kv_pool, block_tables, context_lens, scale, k_scale, v_scale, kv_format="e4m3", out=None,
                  workspace=None, err=None, stream=None):
    """Decode over the 8-bit cache (see include/pa.h)."""
    _need_cuda("q", q)
    _need_cuda("block_tables", block_tables, torch.int32)
    _need_cuda("context_lens", context_lens, torch.int32)
    NB, Hkv, B, d = _need_pool8(kv_pool)
    N, Hq, dq = q.shape
    if dq != d or block_tables.shape[0] != N:
        raise ValueError("q [N, Hq, d] and kv_pool [NB, Hkv, 2, B, d] disagree")
    out = torch.empty_like(q) if out is None else out
    fmt = KV_FORMATS[kv_format]
    shape = make_shape(N, Hq, Hkv, d, B, NB, block_tables.shape[1], q.dtype)
    lib = _lib.load()
    with torch.cuda.device(q.device):
        if workspace is None:
            need = int(lib.pa_decode_fp8_workspace_bytes(ctypes.byref(shape), fmt))
            workspace = _shared_workspace(q.device, max(need, 1), stream)
        st = lib.pa_decode_fp8(ctypes.byref(shape), fmt, _ptr(q), _ptr(kv_pool), _ptr(block_tables),
                               _ptr(context_lens), ctypes.c_float(scale), ctypes.c_float(k_scale),
                               ctypes.c_float(v_scale), _ptr(out), _ptr(workspace),
                               ctypes.c_size_t(workspace.numel() * workspace.element_size()), _ptr(err),
                               _stream(q.device, stream))
    _lib.check(st, "pa_decode_fp8")
    return out


def pa_append_kv_fp8(k_new, v_new, slot_mapping, kv_pool, k_scale, v_scale, kv_format="e4m3", err=None,
                     stream=None):
    """Quantize k_new / v_new [T, Hkv, d] (fp16/bf16) into the 8-bit pool."""
    _need_cuda("k_new", k_new)
    _need_cuda("v_new", v_new, k_new.dtype)
    _need_cuda("slot_mapping", slot_mapping, torch.int64)
    NB, Hkv, B, d = _need_pool8(kv_pool)
    T = slot_mapping.shape[0]
    shape = make_shape(0, 1, Hkv, d, B, NB, 1, k_new.dtype)
    with torch.cuda.device(kv_pool.device):
        st = _lib.load().pa_append_kv_fp8(ctypes.byref(shape), KV_FORMATS[kv_format], ctypes.c_int32(T),
                                          _ptr(k_new), _ptr(v_new), _ptr(slot_mapping), _ptr(kv_pool),
                                          ctypes.c_float(k_scale), ctypes.c_float(v_scale), _ptr(err),
                                          _stream(kv_pool.device, stream))
    _lib.check(st, "pa_append_kv_fp8")


def pa_copy_blocks_fp8(src_dst_pairs, kv_pool, kv_format="e4m3", err=None, stream=None):
    """Copy-on-write copies of whole blocks of the 8-bit pool."""
    _need_cuda("src_dst_pairs", src_dst_pairs, torch.int32)
    NB, Hkv, B, d = _need_pool8(kv_pool)
    shape = _lib.PaShape(0, 1, Hkv, d, B, NB, 1, KV_FORMATS[kv_format])
    with torch.cuda.device(kv_pool.device):
        st = _lib.load().pa_copy_blocks_fp8(ctypes.byref(shape), _ptr(src_dst_pairs),
                                            ctypes.c_int32(src_dst_pairs.shape[0]), _ptr(kv_pool), _ptr(err),
                                            _stream(kv_pool.device, stream))
    _lib.check(st, "pa_copy_blocks_fp8")


# --------------------------------------------------------------------------- 4-bit cache
def int4_pool(num_blocks, num_kv_heads, block_size, head_dim=128, device="cuda"):
    """A zeroed 4-bit pool.  Its tensor shape [NB, Hkv, B, d + 8] only sizes
    the bytes of each (block, head) piece (B * d code nibbles + 8 * B scale
    bytes); the piece layout itself is the one include/pa.h describes."""
    return torch.zeros((num_blocks, num_kv_heads, block_size, head_dim + 8), dtype=torch.uint8, device=device)


def _need_pool4(kv_pool):
    _need_cuda("kv_pool", kv_pool, torch.uint8)
    if kv_pool.dim() != 4:
        raise ValueError("kv_pool must be uint8 [NB, Hkv, B, d + 8] (see int4_pool)")
    return kv_pool.shape[0], kv_pool.shape[1], kv_pool.shape[2], kv_pool.shape[3] - 8


def pa_decode_int4(q, kv_pool, block_tables, context_lens, scale, out=None, workspace=None, err=None,
                   stream=None):
    """Decode over the 4-bit cache (see include/pa.h)."""
    _need_cuda("q", q)
    _need_cuda("block_tables", block_tables, torch.int32)
    _need_cuda("context_lens", context_lens, torch.int32)
    NB, Hkv, B, d = _need_pool4(kv_pool)
    N, Hq, dq = q.shape
    if dq != d or block_tables.shape[0] != N:
        raise ValueError("q [N, Hq, d] and kv_pool [NB, Hkv, B, d + 8] disagree")
    out = torch.empty_like(q) if out is None else out
    shape = make_shape(N, Hq, Hkv, d, B, NB, block_tables.shape[1], q.dtype)
    lib = _lib.load()
    with torch.cuda.device(q.device):
        if workspace is None:
            need = int(lib.pa_decode_int4_workspace_bytes(ctypes.byref(shape)))
            workspace = _shared_workspace(q.device, max(need, 1), stream)
        st = lib.pa_decode_int4(ctypes.byref(shape), _ptr(q), _ptr(kv_pool), _ptr(block_tables),
                                _ptr(context_lens), ctypes.c_float(scale), _ptr(out), _ptr(workspace),
                                ctypes.c_size_t(workspace.numel() * workspace.element_size()), _ptr(err),
                                _stream(q.device, stream))
    _lib.check(st, "pa_decode_int4")
    return out


def pa_append_kv_int4(k_new, v_new, slot_mapping, kv_pool, err=None, stream=None):
    """Quantize k_new / v_new [T, Hkv, d] (fp16/bf16) into the 4-bit pool."""
    _need_cuda("k_new", k_new)
    _need_cuda("v_new", v_new, k_new.dtype)
    _need_cuda("slot_mapping", slot_mapping, torch.int64)
    NB, Hkv, B, d = _need_pool4(kv_pool)
    T = slot_mapping.shape[0]
    shape = make_shape(0, 1, Hkv, d, B, NB, 1, k_new.dtype)
    with torch.cuda.device(kv_pool.device):
        st = _lib.load().pa_append_kv_int4(ctypes.byref(shape), ctypes.c_int32(T), _ptr(k_new), _ptr(v_new),
                                           _ptr(slot_mapping), _ptr(kv_pool), _ptr(err),
                                           _stream(kv_pool.device, stream))
    _lib.check(st, "pa_append_kv_int4")


def pa_copy_blocks_int4(src_dst_pairs, kv_pool, dtype=torch.bfloat16, err=None, stream=None):
    """Copy-on-write copies of whole blocks of the 4-bit pool."""
    _need_cuda("src_dst_pairs", src_dst_pairs, torch.int32)
    NB, Hkv, B, d = _need_pool4(kv_pool)
    shape = make_shape(0, 1, Hkv, d, B, NB, 1, dtype)
    with torch.cuda.device(kv_pool.device):
        st = _lib.load().pa_copy_blocks_int4(ctypes.byref(shape), _ptr(src_dst_pairs),
                                             ctypes.c_int32(src_dst_pairs.shape[0]), _ptr(kv_pool), _ptr(err),
                                             _stream(kv_pool.device, stream))
    _lib.check(st, "pa_copy_blocks_int4")
