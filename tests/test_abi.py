"""The C ABI library builds, loads and exports what include/pa.h declares;
host-side argument checks answer without touching a GPU."""

import ctypes
import os
import re

import pytest

from paged_kv_cache_254_gb300 import _build, _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return _lib.load()


def header_functions():
    text = open(os.path.join(ROOT, "include", "pa.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pa_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    declared = header_functions()
    assert set(declared) == set(_lib.EXPORTS)
    for name in declared:
        assert hasattr(lib, name), name


def test_version_and_status_strings(lib):
    assert lib.pa_version() == 100
    for code in range(7):
        assert lib.pa_status_string(code).decode() not in ("", "unknown status")
    assert lib.pa_status_string(99).decode() == "unknown status"


def shape(**kw):
    base = dict(num_seqs=4, num_q_heads=8, num_kv_heads=8, head_dim=64, block_size=16, num_blocks=64,
                max_blocks_per_seq=7, dtype=_lib.PA_FP16)
    base.update(kw)
    return _lib.PaShape(*[base[f] for f, _ in _lib.PaShape._fields_])


NULL = ctypes.c_void_p(0)
BUF_BYTES = 1 << 20
_bufs = []


def _real_buffer(nbytes=BUF_BYTES):
    """Real, zeroed, 256-byte aligned memory for the pointer arguments whose
    checks these tests exercise.  With a GPU present it is device memory, so a
    host check that regressed would send a kernel to valid memory of the size
    the call is told, never to an unmapped address; without one it is host
    memory (no kernel can launch)."""
    try:
        import torch
        cuda = torch.cuda.is_available()
    except Exception:   # pragma: no cover
        cuda = False
    if cuda:
        t = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
        _bufs.append(t)
        return ctypes.c_void_p(t.data_ptr())
    b = (ctypes.c_uint8 * (nbytes + 256))()
    _bufs.append(b)
    return ctypes.c_void_p((ctypes.addressof(b) + 255) & ~255)


FAKE = _real_buffer()   # every pointer argument that must pass the null check


def decode_status(lib, s, q=FAKE, scale=0.125, ws=FAKE, ws_bytes=BUF_BYTES):
    return lib.pa_decode(ctypes.byref(s), q, FAKE, FAKE, FAKE, FAKE, ctypes.c_float(scale), FAKE, ws,
                         ctypes.c_size_t(ws_bytes), NULL, NULL)


@pytest.mark.parametrize("kw,status", [
    (dict(num_q_heads=12, num_kv_heads=8), 1),      # Hq % Hkv != 0
    (dict(num_kv_heads=0), 1),
    (dict(num_seqs=-1), 1),
    (dict(dtype=7), 1),
    (dict(head_dim=96), 2),
    (dict(block_size=8), 2),
    (dict(num_q_heads=24, num_kv_heads=8), 2),      # group of 3
    (dict(num_q_heads=64, num_kv_heads=2), 2),      # group of 32
    (dict(num_blocks=1 << 26, num_kv_heads=8, num_q_heads=8), 2),   # pool rows >= 2^31
])
def test_decode_rejects_bad_shapes(lib, kw, status):
    assert decode_status(lib, shape(**kw)) == status


def test_decode_rejects_null_and_misaligned(lib):
    s = shape()
    assert decode_status(lib, s, q=NULL) == 1
    assert decode_status(lib, s, q=ctypes.c_void_p(FAKE.value + 2)) == 1
    assert decode_status(lib, s, scale=float("nan")) == 1
    assert lib.pa_decode(None, FAKE, FAKE, FAKE, FAKE, FAKE, ctypes.c_float(1.0), FAKE, FAKE, 0, NULL, NULL) == 1


def test_empty_batch_is_a_no_op(lib):
    assert decode_status(lib, shape(num_seqs=0)) == 0


def test_append_and_copy_checks(lib):
    s = shape()
    assert lib.pa_append_kv(ctypes.byref(s), -1, FAKE, FAKE, FAKE, FAKE, FAKE, NULL, NULL) == 1
    assert lib.pa_append_kv(ctypes.byref(s), 0, NULL, NULL, NULL, NULL, NULL, NULL, NULL) == 0
    assert lib.pa_append_kv(ctypes.byref(s), 3, NULL, FAKE, FAKE, FAKE, FAKE, NULL, NULL) == 1
    assert lib.pa_copy_blocks(ctypes.byref(s), FAKE, -2, FAKE, FAKE, NULL, NULL) == 1
    assert lib.pa_copy_blocks(ctypes.byref(s), NULL, 0, NULL, NULL, NULL, NULL) == 0
    assert lib.pa_copy_blocks(ctypes.byref(s), NULL, 4, FAKE, FAKE, NULL, NULL) == 1
    bad = shape(dtype=7)
    assert lib.pa_copy_blocks(ctypes.byref(bad), FAKE, 1, FAKE, FAKE, NULL, NULL) == 1
    assert lib.pa_read_error(NULL, NULL) == 1


def test_workspace_query_rejects_bad_shape(lib):
    assert lib.pa_decode_workspace_bytes(ctypes.byref(shape(head_dim=80))) == 0
    assert lib.pa_decode_workspace_bytes(None) == 0


def test_product_path_fails_loudly_without_library(monkeypatch):
    monkeypatch.setattr(_lib, "_lib", None)
    monkeypatch.setattr(_lib, "library_path", lambda: "/nonexistent/libpa.so")
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        _lib.load()


def test_fp8_entry_point_checks(lib):
    s = shape(head_dim=128, num_q_heads=8, num_kv_heads=2)
    f = ctypes.c_float

    def dec(sh, fmt=2, ks=1.0, vs=1.0, q=FAKE):
        return lib.pa_decode_fp8(ctypes.byref(sh), fmt, q, FAKE, FAKE, FAKE, f(0.1), f(ks), f(vs), FAKE,
                                 FAKE, ctypes.c_size_t(BUF_BYTES), NULL, NULL)
    assert dec(s, fmt=0) == 1                      # a 16-bit code is not an 8-bit format
    assert dec(s, ks=0.0) == 1 and dec(s, vs=float("inf")) == 1
    assert dec(shape(head_dim=64)) == 2            # 8-bit cache rows must be 128 bytes
    assert dec(shape(head_dim=128, dtype=2)) == 1  # queries must be 16-bit
    assert dec(s, q=NULL) == 1
    assert dec(shape(head_dim=128, num_seqs=0)) == 0

    def app(sh, fmt=2, n=4, ks=1.0):
        return lib.pa_append_kv_fp8(ctypes.byref(sh), fmt, n, FAKE, FAKE, FAKE, FAKE, f(ks), f(1.0), NULL, NULL)
    assert app(s, fmt=5) == 1 and app(s, ks=-1.0) == 1 and app(s, n=-1) == 1
    assert app(shape(head_dim=128, dtype=3)) == 1  # new values must be 16-bit
    assert app(s, n=0) == 0
    # 16-bit entry points refuse an 8-bit dtype
    assert lib.pa_append_kv(ctypes.byref(shape(dtype=2)), 1, FAKE, FAKE, FAKE, FAKE, FAKE, NULL, NULL) == 1
    assert decode_status(lib, shape(dtype=2)) == 1
    # whole-block copies of the 8-bit pool take its format as shape->dtype
    assert lib.pa_copy_blocks_fp8(ctypes.byref(shape(dtype=1)), FAKE, 1, FAKE, NULL, NULL) == 1
    assert lib.pa_copy_blocks_fp8(ctypes.byref(shape(dtype=2)), FAKE, -1, FAKE, NULL, NULL) == 1
    assert lib.pa_copy_blocks_fp8(ctypes.byref(shape(dtype=2)), NULL, 0, NULL, NULL, NULL) == 0
    assert lib.pa_copy_blocks(ctypes.byref(shape(dtype=2)), FAKE, 1, FAKE, FAKE, NULL, NULL) == 1


def test_int4_entry_point_checks(lib):
    s = shape(head_dim=128, num_q_heads=8, num_kv_heads=2)
    f = ctypes.c_float

    def dec(sh, q=FAKE, scale=0.1):
        return lib.pa_decode_int4(ctypes.byref(sh), q, FAKE, FAKE, FAKE, f(scale), FAKE, FAKE,
                                  ctypes.c_size_t(BUF_BYTES), NULL, NULL)
    assert dec(shape(head_dim=64)) == 2                     # the 4-bit layout is for head_dim 128
    assert dec(shape(head_dim=128, block_size=8)) == 2
    assert dec(s, q=NULL) == 1 and dec(s, scale=float("nan")) == 1
    assert dec(shape(head_dim=128, num_seqs=0)) == 0
    assert lib.pa_append_kv_int4(ctypes.byref(s), -1, FAKE, FAKE, FAKE, FAKE, NULL, NULL) == 1
    assert lib.pa_append_kv_int4(ctypes.byref(s), 0, NULL, NULL, NULL, NULL, NULL, NULL) == 0
    assert lib.pa_append_kv_int4(ctypes.byref(s), 3, NULL, FAKE, FAKE, FAKE, NULL, NULL) == 1
    assert lib.pa_append_kv_int4(ctypes.byref(shape(head_dim=64)), 3, FAKE, FAKE, FAKE, FAKE, NULL, NULL) == 2
    assert lib.pa_copy_blocks_int4(ctypes.byref(s), FAKE, -1, FAKE, NULL, NULL) == 1
    assert lib.pa_copy_blocks_int4(ctypes.byref(s), NULL, 0, NULL, NULL, NULL) == 0
    assert lib.pa_copy_blocks_int4(ctypes.byref(s), NULL, 2, FAKE, NULL, NULL) == 1
    assert lib.pa_decode_int4_workspace_bytes(ctypes.byref(shape(head_dim=64))) == 0


def test_multi_token_entry_point_checks(lib):
    s = shape(head_dim=128, num_q_heads=8, num_kv_heads=2)

    def dec(sh, max_q=4, total=8, q=FAKE, q_start=FAKE, scale=0.1):
        return lib.pa_decode_multi(ctypes.byref(sh), max_q, total, q, q_start, FAKE, FAKE, FAKE, FAKE,
                                   ctypes.c_float(scale), FAKE, FAKE, ctypes.c_size_t(BUF_BYTES), NULL, NULL)
    assert dec(s, max_q=0) == 1 and dec(s, max_q=17) == 1     # chunks of 1..16 tokens
    assert dec(shape(head_dim=128, num_q_heads=32, num_kv_heads=2), max_q=16) == 2   # 256 rows per pair
    assert dec(s, total=-1) == 1
    assert dec(s, q_start=NULL) == 1
    assert dec(s, q=NULL) == 1                                  # rows to compute but no q
    assert dec(s, scale=float("inf")) == 1
    assert dec(shape(head_dim=128, num_q_heads=8, num_kv_heads=2, num_seqs=0)) == 0
    assert dec(shape(head_dim=96)) == 2
    assert lib.pa_decode_multi_workspace_bytes(ctypes.byref(s), 0) == 0


def test_shared_prefix_and_noalloc_checks(lib):
    s = shape(head_dim=128, num_q_heads=8, num_kv_heads=2)

    def dec(sh, groups=1, starts=FAKE, prefix=FAKE):
        return lib.pa_decode_shared_prefix(ctypes.byref(sh), FAKE, FAKE, FAKE, FAKE, FAKE, groups, starts, prefix,
                                           ctypes.c_float(0.1), FAKE, FAKE, ctypes.c_size_t(BUF_BYTES), NULL, NULL)
    assert dec(s, groups=-1) == 1
    assert dec(s, groups=2, starts=NULL) == 1 and dec(s, groups=2, prefix=NULL) == 1
    assert dec(shape(head_dim=128, num_q_heads=8, num_kv_heads=2, num_seqs=0)) == 0
    assert dec(shape(num_q_heads=12, num_kv_heads=8)) == 1
    assert lib.pa_decode_shared_prefix_workspace_bytes(ctypes.byref(shape(block_size=8))) == 0
    # a shape no decode kernel serves is refused before any scratch is touched
    assert lib.pa_decode_noalloc(ctypes.byref(shape(head_dim=96)), NULL, NULL, NULL, NULL, NULL,
                                 ctypes.c_float(0.1), NULL, NULL, NULL) == 2
    assert lib.pa_decode_noalloc(ctypes.byref(shape(num_q_heads=12, num_kv_heads=8)), NULL, NULL, NULL, NULL,
                                 NULL, ctypes.c_float(0.1), NULL, NULL, NULL) == 1


def test_stall_setter_checks_its_limit(lib):
    assert lib.pa_set_decode_stall_ns(2_000_000_000) == 1   # above one second
    assert lib.pa_set_decode_stall_ns(0) == 0
