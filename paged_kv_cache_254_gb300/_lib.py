"""ctypes binding of libpa.so (argument marshalling only).

Every computation runs in the library's CUDA kernels; this module only turns
torch tensors into pointers, shapes and the current stream, and status codes
into exceptions.  If the library has not been built it raises at once: there
is no fallback path.
"""

from __future__ import annotations

import ctypes
import os
import threading

from . import _build

PA_OK = 0
STATUS_NAMES = {
    0: "PA_OK", 1: "PA_ERR_INVALID_ARG", 2: "PA_ERR_UNSUPPORTED", 3: "PA_ERR_CUDA",
    4: "PA_ERR_OUT_OF_RANGE", 5: "PA_ERR_TIMEOUT", 6: "PA_ERR_WORKSPACE",
}
PA_FP16, PA_BF16, PA_FP8_E4M3, PA_FP8_E5M2 = 0, 1, 2, 3
DEVERR_BLOCK_ID, DEVERR_CONTEXT, DEVERR_SLOT, DEVERR_COPY_PAIR, DEVERR_TIMEOUT, DEVERR_GROUP = 1, 2, 4, 8, 16, 32
DEVERR_Q_RANGE = 64

# Every symbol include/pa.h declares.
EXPORTS = ("pa_decode_workspace_bytes", "pa_decode", "pa_append_kv", "pa_copy_blocks", "pa_read_error",
           "pa_status_string", "pa_version", "pa_decode_noalloc", "pa_decode_shared_prefix_workspace_bytes",
           "pa_decode_shared_prefix", "pa_decode_fp8_workspace_bytes", "pa_decode_fp8", "pa_append_kv_fp8",
           "pa_copy_blocks_fp8", "pa_decode_multi_workspace_bytes", "pa_decode_multi",
           "pa_decode_int4_workspace_bytes", "pa_decode_int4", "pa_append_kv_int4", "pa_copy_blocks_int4",
           "pa_set_decode_stall_ns")
NOALLOC_SCRATCH_BYTES = 32 << 20


class PaShape(ctypes.Structure):
    _fields_ = [
        ("num_seqs", ctypes.c_int32),
        ("num_q_heads", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("block_size", ctypes.c_int32),
        ("num_blocks", ctypes.c_int32),
        ("max_blocks_per_seq", ctypes.c_int32),
        ("dtype", ctypes.c_int32),
    ]


class PagedAttentionError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {STATUS_NAMES.get(status, status)} ({status_string(status)})")


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _build.LIBPATH


def load() -> ctypes.CDLL:
    """Load libpa.so (built by ``_build.build()``); raise if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(f"libpa.so is not built ({path}); run paged_kv_cache_254_gb300._build.build() "
                               "with the CUDA toolkit first -- there is no CPU fallback")
        lib = ctypes.CDLL(path)
        P, I32, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
        SP = ctypes.POINTER(PaShape)
        lib.pa_decode_workspace_bytes.argtypes = [SP]
        lib.pa_decode_workspace_bytes.restype = SZ
        lib.pa_decode.argtypes = [SP, P, P, P, P, P, ctypes.c_float, P, P, SZ, P, P]
        lib.pa_decode.restype = I32
        lib.pa_append_kv.argtypes = [SP, I32, P, P, P, P, P, P, P]
        lib.pa_append_kv.restype = I32
        lib.pa_copy_blocks.argtypes = [SP, P, I32, P, P, P, P]
        lib.pa_copy_blocks.restype = I32
        lib.pa_read_error.argtypes = [P, P]
        lib.pa_read_error.restype = I32
        lib.pa_status_string.argtypes = [I32]
        lib.pa_status_string.restype = ctypes.c_char_p
        lib.pa_version.argtypes = []
        lib.pa_version.restype = I32
        lib.pa_decode_noalloc.argtypes = [SP, P, P, P, P, P, ctypes.c_float, P, P, P]
        lib.pa_decode_noalloc.restype = I32
        lib.pa_decode_shared_prefix_workspace_bytes.argtypes = [SP]
        lib.pa_decode_shared_prefix_workspace_bytes.restype = SZ
        lib.pa_decode_shared_prefix.argtypes = [SP, P, P, P, P, P, I32, P, P, ctypes.c_float, P, P, SZ, P, P]
        lib.pa_decode_shared_prefix.restype = I32
        F = ctypes.c_float
        lib.pa_decode_fp8_workspace_bytes.argtypes = [SP, I32]
        lib.pa_decode_fp8_workspace_bytes.restype = SZ
        lib.pa_decode_fp8.argtypes = [SP, I32, P, P, P, P, F, F, F, P, P, SZ, P, P]
        lib.pa_decode_fp8.restype = I32
        lib.pa_append_kv_fp8.argtypes = [SP, I32, I32, P, P, P, P, F, F, P, P]
        lib.pa_append_kv_fp8.restype = I32
        lib.pa_copy_blocks_fp8.argtypes = [SP, P, I32, P, P, P]
        lib.pa_copy_blocks_fp8.restype = I32
        lib.pa_decode_multi_workspace_bytes.argtypes = [SP, I32]
        lib.pa_decode_multi_workspace_bytes.restype = SZ
        lib.pa_decode_multi.argtypes = [SP, I32, I32, P, P, P, P, P, P, ctypes.c_float, P, P, SZ, P, P]
        lib.pa_decode_multi.restype = I32
        lib.pa_decode_int4_workspace_bytes.argtypes = [SP]
        lib.pa_decode_int4_workspace_bytes.restype = SZ
        lib.pa_decode_int4.argtypes = [SP, P, P, P, P, ctypes.c_float, P, P, SZ, P, P]
        lib.pa_decode_int4.restype = I32
        lib.pa_append_kv_int4.argtypes = [SP, I32, P, P, P, P, P, P]
        lib.pa_append_kv_int4.restype = I32
        lib.pa_copy_blocks_int4.argtypes = [SP, P, I32, P, P, P]
        lib.pa_copy_blocks_int4.restype = I32
        lib.pa_set_decode_stall_ns.argtypes = [ctypes.c_uint64]
        lib.pa_set_decode_stall_ns.restype = I32
        _lib = lib
        return lib


def status_string(status: int) -> str:
    try:
        return load().pa_status_string(int(status)).decode()
    except Exception:  # pragma: no cover - only used for messages
        return "?"


def check(status: int, what: str) -> None:
    if status != PA_OK:
        raise PagedAttentionError(status, what)
