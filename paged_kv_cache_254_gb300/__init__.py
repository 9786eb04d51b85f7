"""Paged KV-cache decode attention for GB300 (sm_103a).

* ``pa_decode``, ``pa_append_kv``, ``pa_copy_blocks``, ``pa_read_error`` --
  thin bindings of the C ABI in ``include/pa.h`` (libpa.so, CUDA kernels).
* ``BlockManager`` -- host bookkeeping that builds block tables, slot
  mappings and copy-on-write copy lists.

The CUDA library is loaded on first use; without it every entry point raises.
"""

from ._lib import PagedAttentionError  # noqa: F401
from .block_manager import BlockManager  # noqa: F401
from .ops import (  # noqa: F401
    make_shape,
    new_error_word,
    pa_append_kv,
    pa_copy_blocks,
    pa_append_kv_fp8,
    pa_copy_blocks_fp8,
    pa_decode,
    pa_decode_fp8,
    pa_decode_shared_prefix,
    pa_decode_multi,
    pa_decode_int4,
    pa_append_kv_int4,
    pa_copy_blocks_int4,
    int4_pool,
    pa_decode_workspace_bytes,
    pa_read_error,
    pa_set_decode_stall_ns,
    workspace_for,
)

__version__ = "0.1.0"
