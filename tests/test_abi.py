"""The C-ABI library loads on a machine without a GPU, exports every symbol its header declares,
and rejects bad arguments on the host before touching a device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dsattn.h")


@pytest.fixture(scope="module")
def lib():
    from sparse_latent_attention_attn_gb300 import build
    path = build.build()
    return ctypes.CDLL(path)


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ds_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("ds_window_topk_idxs", "ds_kv_quant_ring_write", "ds_sparse_attn",
                     "ds_sparse_attn_workspace_bytes", "ds_device_status", "ds_status_string",
                     "ds_kv_quantize_fp8", "ds_kv_quant_ring_write_fp8", "ds_sparse_attn_fp8kv",
                     "ds_apply_rotary", "ds_kv_rope_quant_ring_write"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    lib.ds_status_string.restype = ctypes.c_char_p
    for code in (0, -1, -2, -3, -4, -5):
        s = lib.ds_status_string(code).decode()
        assert s and s != "unknown status"
    assert lib.ds_status_string(12345).decode() == "unknown status"


def test_host_side_argument_checks(lib):
    P = ctypes.c_void_p
    f = lib.ds_sparse_attn
    f.argtypes = [P, P, ctypes.c_int64, P, P, ctypes.c_int, ctypes.c_float, P, ctypes.c_int, ctypes.c_int,
                  ctypes.c_int, ctypes.c_int, P, ctypes.c_size_t, P]
    fake = P(4096)   # never dereferenced: every call below fails its checks first
    # unsupported head_dim / head count
    assert f(fake, fake, 10, fake, fake, 4, 0.1, fake, 1, 1, 4, 48, None, 0, None) == -2
    assert f(fake, fake, 10, fake, fake, 4, 0.1, fake, 1, 1, 129, 64, None, 0, None) == -2
    # null pointers, negative sizes, zero heads
    assert f(None, fake, 10, fake, fake, 4, 0.1, fake, 1, 1, 4, 64, None, 0, None) == -1
    assert f(fake, fake, 10, fake, fake, -1, 0.1, fake, 1, 1, 4, 64, None, 0, None) == -1
    assert f(fake, fake, 10, fake, fake, 4, 0.1, fake, 1, 1, 0, 64, None, 0, None) == -1
    # misaligned q
    assert f(P(4097), fake, 10, fake, fake, 4, 0.1, fake, 1, 1, 4, 64, None, 0, None) == -1
    # nothing to do is not an error
    assert f(None, None, 0, None, None, 0, 0.1, None, 0, 1, 4, 64, None, 0, None) == 0

    w = lib.ds_window_topk_idxs
    w.argtypes = [P, ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_int64, ctypes.c_int,
                  ctypes.POINTER(ctypes.c_int), P]
    assert w(None, 8, 1, 4, 0, 8, None, None) == -1
    assert w(fake, 8, 1, 4, 5, 8, None, None) == -2           # chunked prefill is not defined
    assert w(fake, 4, 1, 12, 0, 8, None, None) == -1          # ld < cols

    q = lib.ds_kv_quant_ring_write
    q.argtypes = [P, ctypes.c_int64, P, ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int64,
                  ctypes.c_int, P]
    assert q(fake, 40, None, 0, 1, 1, 40, 0, 8, None) == -1   # d not a multiple of 32
    assert q(None, 64, None, 0, 1, 1, 64, 0, 8, None) == -1
    assert q(P(4104), 64, None, 0, 1, 1, 64, 0, 8, None) == -1  # misaligned


def test_fp8_store_argument_checks(lib):
    P = ctypes.c_void_p
    fake = P(4096)   # never dereferenced: every call below fails its checks first
    z = lib.ds_kv_quantize_fp8
    z.argtypes = [P, ctypes.c_int64, ctypes.c_int, P, P, P]
    assert z(fake, 4, 40, fake, fake, None) == -1             # d not a multiple of 32
    assert z(None, 4, 64, fake, fake, None) == -1
    assert z(fake, 4, 64, P(4100), fake, None) == -1          # misaligned codes
    assert z(None, 0, 64, None, None, None) == 0              # nothing to do
    r = lib.ds_kv_quant_ring_write_fp8
    r.argtypes = [P, ctypes.c_int64, P, P, ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                  ctypes.c_int64, ctypes.c_int, P]
    assert r(fake, 64, fake, fake, 7, 1, 1, 64, 0, 8, None) == -1     # ring rows < window
    assert r(fake, 64, None, fake, 8, 1, 1, 64, 0, 8, None) == -1
    f = lib.ds_sparse_attn_fp8kv
    f.argtypes = [P, P, P, ctypes.c_int64, P, P, ctypes.c_int, ctypes.c_float, P, ctypes.c_int, ctypes.c_int,
                  ctypes.c_int, ctypes.c_int, P, ctypes.c_size_t, P]
    assert f(fake, fake, fake, 10, fake, fake, 4, 0.1, fake, 1, 1, 4, 64, None, 0, None) == -2   # d = 512 only
    assert f(fake, None, fake, 10, fake, fake, 4, 0.1, fake, 1, 1, 4, 512, None, 0, None) == -1
    assert f(fake, fake, None, 10, fake, fake, 4, 0.1, fake, 1, 1, 4, 512, None, 0, None) == -1
    assert f(fake, P(4104), fake, 10, fake, fake, 4, 0.1, fake, 1, 1, 4, 512, None, 0, None) == -1


def test_rope_argument_checks(lib):
    P = ctypes.c_void_p
    fake = P(4096)
    r = lib.ds_apply_rotary
    r.argtypes = [P, ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, P,
                  ctypes.c_int64, ctypes.c_int, P]
    assert r(fake, 4, 64, 12, 1, 1, 0, fake, 10, 0, None) == -1     # rd not a multiple of 8
    assert r(fake, 4, 64, 128, 1, 1, 0, fake, 10, 0, None) == -1    # rd > row_len
    assert r(fake, 9, 64, 32, 3, 3, 8, fake, 10, 0, None) == -1     # rows at positions 8, 9, 10: 10 is past the table
    assert r(None, 4, 64, 32, 1, 1, 0, fake, 10, 0, None) == -1
    assert r(fake, 0, 64, 32, 1, 1, 0, fake, 10, 0, None) == 0      # nothing to do
    k = lib.ds_kv_rope_quant_ring_write
    k.argtypes = [P, ctypes.c_int64, P, ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int64,
                  ctypes.c_int, ctypes.c_int, P, ctypes.c_int64, P]
    assert k(fake, 64, None, 0, 1, 1, 64, 0, 8, 48, fake, 10, None) == -1   # rd not whole blocks
    assert k(fake, 64, None, 0, 1, 1, 64, 10, 8, 32, fake, 10, None) == -1  # position 10 outside the table
    assert k(fake, 64, None, 0, 1, 1, 64, 0, 8, 32, None, 10, None) == -1


def test_sparse_attn_rope_argument_checks(lib):
    P = ctypes.c_void_p
    fake = P(4096)   # never dereferenced: every call below fails its checks first
    f = lib.ds_sparse_attn_rope
    f.argtypes = [P, P, ctypes.c_int64, P, P, ctypes.c_int, ctypes.c_float, P, ctypes.c_int, ctypes.c_int,
                  ctypes.c_int, ctypes.c_int, P, ctypes.c_size_t, ctypes.c_int, P, ctypes.c_int64, ctypes.c_int64, P]
    args = lambda rd, table, rows, pos, m=1: (fake, fake, 10, fake, fake, 4, 0.1, fake, 1, m, 4, 64, None, 0, rd,
                                               table, rows, pos, None)
    assert f(*args(12, fake, 100, 0)) == -1          # rd not a multiple of 8
    assert f(*args(128, fake, 100, 0)) == -1         # rd > d
    assert f(*args(16, None, 100, 0)) == -1          # no table
    assert f(*args(16, P(4100), 100, 0)) == -1       # table not 8-byte aligned
    assert f(*args(16, fake, 100, 98, m=3)) == -1    # positions 98..100: 100 is past the table
    assert f(*args(16, fake, 100, -1)) == -1


def test_workspace_query_is_host_only(lib):
    f = lib.ds_sparse_attn_workspace_bytes
    f.argtypes = [ctypes.c_int] * 5
    f.restype = ctypes.c_size_t
    assert f(1, 1, 4, 48, 8) == 0          # unsupported shapes need nothing
    assert f(1, 1, 129, 64, 8) == 0
