"""The C ABI library: it builds, loads, exports what include/*.h declares, and its host-side
validation rejects bad calls before anything is enqueued (no GPU needed)."""

import ctypes
import os
import re

import pytest

import oracle as O

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from looped_transformer_kv_gb300 import build
    build.build()
    from looped_transformer_kv_gb300 import _lib
    return _lib


def _declared():
    names = []
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            src = open(os.path.join(ROOT, "include", f)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names += re.findall(r"\b(rq_[a-z0-9_]+)\s*\(", src)
    return sorted(set(names))


def test_every_declared_symbol_is_exported(lib):
    L = lib.lib()
    declared = _declared()
    assert {"rq_encode_append", "rq_decode_attention", "rq_bf16_decode_attention"} <= set(declared)
    for n in declared:
        assert hasattr(L, n), n
    assert set(lib.EXPORTS) == set(declared)


def _shape(lib, **kw):
    from looped_transformer_kv_gb300 import rq
    a = dict(batch=2, n_q_heads=4, n_kv_heads=2, head_dim=128, n_loops=4, capacity=64,
             res_bits=(2, 2, 2))
    a.update(kw)
    return rq.make_shape(**a)


@pytest.mark.parametrize("d,L,bits", [(128, 4, (2, 2, 2)), (64, 4, (4, 2, 2)), (128, 8, (2,) * 7),
                                      (128, 1, ())])
def test_cache_bytes_closed_form(lib, d, L, bits):
    s = _shape(lib, head_dim=d, n_loops=L, res_bits=bits)
    assert lib.lib().rq_cache_bytes(ctypes.byref(s)) == O.cache_bytes(d, L, bits, 64, 2, 2)


@pytest.mark.parametrize("d,L,bits", [(128, 4, (2, 2, 2)), (64, 4, (4, 2, 2)), (128, 1, ())])
def test_record_bytes_is_64_token_heads(lib, d, L, bits):
    s = _shape(lib, head_dim=d, n_loops=L, res_bits=bits)
    assert lib.lib().rq_record_bytes(ctypes.byref(s)) == O.cache_bytes(d, L, bits, 64)


def test_misaligned_records_are_rejected(lib):
    L = lib.lib()
    s = _shape(lib)
    c = lib.RqCache()
    c.data = 256 + 8                                            # not 16-byte aligned
    c.rot_signs[0] = c.rot_signs[1] = 16
    p = ctypes.c_void_p(16)
    assert L.rq_decode_attention(ctypes.byref(s), ctypes.byref(c), p, 0, 1, None, p, 64, p, p,
                                 1 << 40, None) == 1


def test_status_strings(lib):
    L = lib.lib()
    assert L.rq_status_str(0) == b"RQ_OK"
    assert L.rq_status_str(3) == b"RQ_ERR_WORKSPACE"


@pytest.mark.parametrize("bad,status", [
    (dict(group=64), 2), (dict(head_dim=96), 2), (dict(res_bits=(3, 2, 2)), 2),
    (dict(n_q_heads=3), 1), (dict(capacity=63), 1), (dict(n_loops=17), 2), (dict(batch=0), 1),
])
def test_invalid_shapes_are_rejected_without_launch(lib, bad, status):
    L = lib.lib()
    s = _shape(lib, **bad)
    c = lib.RqCache()
    st = (ctypes.c_int64 * 5)(0, 0, 0, 0, 0)
    # non-null dummies: validation must fail on the shape before any pointer is used
    r = L.rq_encode_append(ctypes.byref(s), ctypes.byref(c), ctypes.c_void_p(16), st, None, 0, 1,
                           None)
    assert r == status
    assert L.rq_cache_bytes(ctypes.byref(s)) == 0


def test_null_pointers_and_ranges_are_rejected(lib):
    L = lib.lib()
    s = _shape(lib)
    c = lib.RqCache()
    st = (ctypes.c_int64 * 5)(0, 0, 0, 0, 0)
    assert L.rq_encode_append(ctypes.byref(s), ctypes.byref(c), ctypes.c_void_p(16), st, None,
                              0, 1, None) == 1             # cache arrays missing
    assert L.rq_decode_attention(ctypes.byref(s), ctypes.byref(c), None, 0, 1, None, None, 0,
                                 None, None, 0, None) == 1
    assert L.rq_bf16_decode_attention(ctypes.byref(s), None, None, None, 0, 1, None, None, 0,
                                      None, None, 0, None) == 1
    assert L.rq_decode_workspace_bytes(ctypes.byref(s), 0, 10) == 0


def test_paging_arguments_are_validated(lib):
    L = lib.lib()
    s = _shape(lib, capacity=128)
    c = lib.RqCache()
    st = (ctypes.c_int64 * 5)(0, 0, 0, 0, 0)
    g = lib.RqPaging()
    g.block_table, g.max_pages, g.n_pages = 16, 2, 8          # non-null dummy table
    # null paging, missing table, capacity != 64 * max_pages, no pages: rejected before any
    # pointer is used (the cache arrays are null too, so the paging check must come first or
    # fail the same way)
    assert L.rq_paged_decode_attention(ctypes.byref(s), ctypes.byref(c), None, None, 0, 1, None,
                                       None, 0, None, None, 0, None) == 1
    assert L.rq_paged_encode_append(ctypes.byref(s), ctypes.byref(c), None, ctypes.c_void_p(16),
                                    st, None, 0, 1, None) == 1
    assert L.rq_paged_cache_bytes(ctypes.byref(s), 0) == 0
    assert L.rq_paged_cache_bytes(ctypes.byref(s), 8) == O.cache_bytes(128, 4, (2, 2, 2), 64, 2, 8)


@pytest.mark.parametrize("lc,ctx", [(1, 4096), (4, 4096), (2, 1), (4, 0)])
def test_decode_workspace_is_header_tickets_and_split_records(lib, lc, ctx):
    # header (256 B: error word), one uint32 ticket per (sequence, query head, loop) rounded to
    # 256 B, then n_splits partial records (m, l, 2 pads, acc_ref[d], acc_res[d]) per column
    s = _shape(lib, capacity=4096)
    ws = lib.lib().rq_decode_workspace_bytes(ctypes.byref(s), lc, ctx)
    cols = 2 * 4 * lc
    tickets = -(-cols * 4 // 256) * 256
    rec = (4 + 2 * 128) * 4
    rest = ws - 256 - tickets
    assert rest > 0 and rest % (cols * rec) == 0, (ws, rest)
    assert rest // (cols * rec) <= max(1, -(-ctx // 64))      # at most one split per 64-token tile


@pytest.mark.parametrize("bad,max_ctx,status", [
    (dict(head_dim=96), 64, 2), (dict(group=64), 64, 2), (dict(res_bits=(3, 2, 2)), 64, 2),
    (dict(n_q_heads=3), 64, 1), ({}, 65, 1),                    # max_ctx above capacity
    (dict(batch=4096, n_q_heads=64, n_kv_heads=64, n_loops=16, res_bits=(2,) * 15,
          capacity=65536), 65537, 1),                           # large shape, max_ctx too big
])
def test_noalloc_entry_point_returns_the_workspace_entry_points_status(lib, bad, max_ctx, status):
    # validation of the no-alloc call is the workspace call's, in the same order: an invalid
    # call gets the same status from both, before any device is touched
    L = lib.lib()
    s = _shape(lib, **bad)
    c = lib.RqCache()
    c.data = 256                                                # non-null dummy records
    c.rot_signs[0] = c.rot_signs[1] = 16
    p = ctypes.c_void_p(16)
    ws_status = L.rq_decode_attention(ctypes.byref(s), ctypes.byref(c), p, 0, 1, None, p, max_ctx,
                                      p, p, 1 << 40, None)
    noalloc_status = L.rq_decode_attention_noalloc(ctypes.byref(s), ctypes.byref(c), p, 0, 1,
                                                   None, p, max_ctx, p, None)
    assert ws_status == noalloc_status == status
