"""Thin PyTorch binding of librq: argument marshalling only.

Every step of encode and decode attention runs in the library's CUDA kernels; PyTorch
provides device memory and the current stream.  Names follow the C ABI (include/rq.h).
"""

import ctypes

import torch

from . import _lib
from ._lib import RQ_MAX_LOOPS, RqCache, RqPaging, RqShape, RqSynthParams, check

GROUP = 32


def _ptr(t):
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def make_shape(batch, n_q_heads, n_kv_heads, head_dim, n_loops, capacity, res_bits,
               softmax_scale=0.0, group=GROUP):
    """rq_shape for one layer; res_bits lists the residual bits of loops 0..L-2."""
    s = RqShape()
    s.batch, s.n_q_heads, s.n_kv_heads = batch, n_q_heads, n_kv_heads
    s.head_dim, s.n_loops, s.group, s.capacity = head_dim, n_loops, group, capacity
    for l, b in enumerate(res_bits):
        s.res_bits[l] = int(b)
    s.softmax_scale = float(softmax_scale)
    return s


def res_bits_of(shape):
    return [int(shape.res_bits[l]) for l in range(shape.n_loops - 1)]


PAGE = 64   # tokens per page of a paged cache


class PackedCache:
    """One layer's packed cache in device memory: the tile records of include/rq.h in one
    buffer (256-byte aligned), [B][Hkv][capacity/64] records, or [n_pages][Hkv] in paged
    form, plus the rotation signs.  record_bytes() is rq_record_bytes; section(...) gives the
    byte range of one kind of row inside a record (for reading the cache back)."""

    def __init__(self, shape, rot_signs, device="cuda", n_pages=None):
        B, H, cap, d = shape.batch, shape.n_kv_heads, shape.capacity, shape.head_dim
        self.n_pages = n_pages
        self.shape = shape
        self.rec = int(_lib.lib().rq_record_bytes(ctypes.byref(shape)))
        assert self.rec > 0
        n_rec = (n_pages * H) if n_pages is not None else (B * H * (cap // PAGE))
        self.data = torch.empty(n_rec * self.rec, dtype=torch.uint8, device=device)
        self.rot_signs = rot_signs.to(device=device, dtype=torch.int8).contiguous()  # [2][H][d]
        assert tuple(self.rot_signs.shape) == (2, H, d)
        c = RqCache()
        c.data = self.data.data_ptr()
        for kv in range(2):
            c.rot_signs[kv] = self.rot_signs[kv].data_ptr()
        self.struct = c

    def records(self):
        """The records as [B][Hkv][capacity/64][rec] (or [n_pages][Hkv][rec] when paged)."""
        s = self.shape
        if self.n_pages is not None:
            return self.data.view(self.n_pages, s.n_kv_heads, self.rec)
        return self.data.view(s.batch, s.n_kv_heads, s.capacity // PAGE, self.rec)

    def section(self, kind, kv, loop=None):
        """(byte offset in a record, row bytes) of one kind of 64 rows: kind in 'codes',
        'meta', 'alpha'; loop None = the reference section."""
        d = self.shape.head_dim
        ng = d // GROUP
        if loop is None:
            base = kv * PAGE * (d // 2 + 4 * ng)
            return {"codes": (base, d // 2), "meta": (base + PAGE * d // 2, 4 * ng)}[kind]
        bits = res_bits_of(self.shape)
        off = PAGE * (d + 8 * ng)
        for b in bits[:loop]:
            off += PAGE * (2 * (d * b // 8) + 8 * ng + 4)
        rb = d * bits[loop] // 8
        base = off + kv * PAGE * (rb + 4 * ng + 2)
        return {"codes": (base, rb), "meta": (base + PAGE * rb, 4 * ng),
                "alpha": (base + PAGE * (rb + 4 * ng), 2)}[kind]

    def tensors(self):
        return [self.data]

    def nbytes(self):
        return self.data.numel()


def cache_bytes(shape):
    return int(_lib.lib().rq_cache_bytes(ctypes.byref(shape)))


def advance_ctx(ctx_lens, n, capacity, stream=None):
    """rq_advance_ctx: ctx_lens[b] += n on the device (capped at capacity)."""
    assert ctx_lens.dtype == torch.int32 and ctx_lens.is_contiguous()
    check("rq_advance_ctx", _lib.lib().rq_advance_ctx(_ptr(ctx_lens), ctx_lens.numel(), int(n),
                                                      int(capacity), _stream(stream)))


def paged_cache_bytes(shape, n_pages):
    return int(_lib.lib().rq_paged_cache_bytes(ctypes.byref(shape), int(n_pages)))


def make_paging(block_table, n_pages):
    """rq_paging for a device int32 block table [B][max_pages] (kept alive by the caller)."""
    assert block_table.dtype == torch.int32 and block_table.dim() == 2
    assert block_table.is_contiguous()
    g = RqPaging()
    g.block_table = block_table.data_ptr()
    g.max_pages = block_table.shape[1]
    g.n_pages = int(n_pages)
    return g


def paged_encode_append(shape, cache, paging, kv_new, positions=None, pos_begin=0, stream=None):
    """rq_paged_encode_append; kv_new as in encode_append."""
    assert kv_new.dtype == torch.bfloat16 and kv_new.dim() == 6 and kv_new.stride(5) == 1
    st = (ctypes.c_int64 * 5)(*[kv_new.stride(i) for i in range(5)])
    check("rq_paged_encode_append", _lib.lib().rq_paged_encode_append(
        ctypes.byref(shape), ctypes.byref(cache.struct), ctypes.byref(paging), _ptr(kv_new), st,
        _ptr(positions), int(pos_begin), int(kv_new.shape[1]), _stream(stream)))


def paged_decode_attention(shape, cache, paging, q, loop_begin, loop_count, pending_kv,
                           ctx_lens, max_ctx, out, ws, stream=None):
    check("rq_paged_decode_attention", _lib.lib().rq_paged_decode_attention(
        ctypes.byref(shape), ctypes.byref(cache.struct), ctypes.byref(paging), _ptr(q),
        int(loop_begin), int(loop_count), _ptr(pending_kv), _ptr(ctx_lens), int(max_ctx),
        _ptr(out), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))


def encode_append(shape, cache, kv_new, positions=None, pos_begin=0, stream=None):
    """kv_new: bf16 [B][n_new][2][L][Hkv][d] (any strides, channel stride 1)."""
    assert kv_new.dtype == torch.bfloat16 and kv_new.dim() == 6 and kv_new.stride(5) == 1
    st = (ctypes.c_int64 * 5)(*[kv_new.stride(i) for i in range(5)])
    n_new = kv_new.shape[1]
    check("rq_encode_append", _lib.lib().rq_encode_append(
        ctypes.byref(shape), ctypes.byref(cache.struct), _ptr(kv_new), st, _ptr(positions),
        int(pos_begin), int(n_new), _stream(stream)))


def ablation_encode_append(shape, cache, kv_new, alpha_mode, positions=None, pos_begin=0,
                           stream=None):
    """rq_ablation_encode_append (include/rq_ablation.h): a_l fixed by alpha_mode
    (0 least squares, 1 one, 2 zero)."""
    assert kv_new.dtype == torch.bfloat16 and kv_new.dim() == 6 and kv_new.stride(5) == 1
    st = (ctypes.c_int64 * 5)(*[kv_new.stride(i) for i in range(5)])
    check("rq_ablation_encode_append", _lib.lib().rq_ablation_encode_append(
        ctypes.byref(shape), ctypes.byref(cache.struct), _ptr(kv_new), st, _ptr(positions),
        int(pos_begin), int(kv_new.shape[1]), int(alpha_mode), _stream(stream)))


def ablation_decode_attention(shape, cache, mode, q, loop, pending_kv, ctx_lens, max_ctx, out, ws,
                              stream=None):
    """rq_ablation_decode_attention: per-loop decode of residual loop `loop` over a cache
    encoded with a = 1 (mode 1) or a = 0 (mode 2)."""
    check("rq_ablation_decode_attention", _lib.lib().rq_ablation_decode_attention(
        ctypes.byref(shape), ctypes.byref(cache.struct), int(mode), _ptr(q), int(loop),
        _ptr(pending_kv), _ptr(ctx_lens), int(max_ctx), _ptr(out), _ptr(ws),
        ws.numel() * ws.element_size(), _stream(stream)))


def decode_workspace_bytes(shape, loop_count, max_ctx):
    return int(_lib.lib().rq_decode_workspace_bytes(ctypes.byref(shape), int(loop_count),
                                                    int(max_ctx)))


def decode_attention(shape, cache, q, loop_begin, loop_count, pending_kv, ctx_lens, max_ctx,
                     out, ws, stream=None):
    check("rq_decode_attention", _lib.lib().rq_decode_attention(
        ctypes.byref(shape), ctypes.byref(cache.struct), _ptr(q), int(loop_begin),
        int(loop_count), _ptr(pending_kv), _ptr(ctx_lens), int(max_ctx), _ptr(out), _ptr(ws),
        ws.numel() * ws.element_size(), _stream(stream)))


def decode_attention_noalloc(shape, cache, q, loop_begin, loop_count, pending_kv, ctx_lens,
                             max_ctx, out, stream=None):
    """rq_decode_attention_noalloc: the library's fixed scratch array instead of a workspace."""
    check("rq_decode_attention_noalloc", _lib.lib().rq_decode_attention_noalloc(
        ctypes.byref(shape), ctypes.byref(cache.struct), _ptr(q), int(loop_begin),
        int(loop_count), _ptr(pending_kv), _ptr(ctx_lens), int(max_ctx), _ptr(out),
        _stream(stream)))


def test_decode_attention_wait_runs_out(shape, cache, q, loop_begin, loop_count, pending_kv,
                                        ctx_lens, max_ctx, out, ws, wait_limit_ns, stream=None):
    """rq_test_decode_attention_wait_runs_out (test hook, include/rq_test.h)."""
    check("rq_test_decode_attention_wait_runs_out",
          _lib.lib().rq_test_decode_attention_wait_runs_out(
              ctypes.byref(shape), ctypes.byref(cache.struct), _ptr(q), int(loop_begin),
              int(loop_count), _ptr(pending_kv), _ptr(ctx_lens), int(max_ctx), _ptr(out), _ptr(ws),
              ws.numel() * ws.element_size(), int(wait_limit_ns), _stream(stream)))


def noalloc_scratch_bytes():
    return int(_lib.lib().rq_decode_noalloc_scratch_bytes())


def bf16_decode_attention(shape, k, v, q, loop_begin, loop_count, pending_kv, ctx_lens, max_ctx,
                          out, ws, stream=None):
    check("rq_bf16_decode_attention", _lib.lib().rq_bf16_decode_attention(
        ctypes.byref(shape), _ptr(k), _ptr(v), _ptr(q), int(loop_begin), int(loop_count),
        _ptr(pending_kv), _ptr(ctx_lens), int(max_ctx), _ptr(out), _ptr(ws),
        ws.numel() * ws.element_size(), _stream(stream)))


def synth_params(seed, layer, head_dim, n_kv_heads, dist, sigma, outlier_mult, outlier_table):
    """rq_synth_params; outlier_table: device int32 [Hkv][2][n] (kept alive by the caller)."""
    p = RqSynthParams()
    p.seed, p.layer, p.head_dim, p.n_kv_heads, p.dist = seed, layer, head_dim, n_kv_heads, dist
    for l, s in enumerate(sigma):
        p.sigma[l] = float(s)
    p.outlier_mult = float(outlier_mult)
    p.n_outliers = int(outlier_table.shape[-1]) if outlier_table is not None else 0
    p.outlier_table = outlier_table.data_ptr() if outlier_table is not None else None
    return p


def synth_states(params, out, strides, b0, nb, t0, nt, l0, nl, stream=None):
    st = (ctypes.c_int64 * 5)(*strides)
    check("rq_synth_states", _lib.lib().rq_synth_states(
        ctypes.byref(params), _ptr(out), st, b0, nb, t0, nt, l0, nl, _stream(stream)))


def synth_queries(params, out, n_q_heads, b0, nb, l0, nl, step=0, stream=None):
    check("rq_synth_queries", _lib.lib().rq_synth_queries(
        ctypes.byref(params), _ptr(out), n_q_heads, b0, nb, l0, nl, step, _stream(stream)))
