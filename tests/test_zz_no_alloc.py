"""rq_decode_attention_noalloc, the entry point for callers that cannot allocate device
memory (a plug-in whose host framework owns all device memory, a C caller that must not
allocate after start-up): it must give the same attention, bit for bit, as
rq_decode_attention with a caller-provided workspace (same kernels, same split plan), on
consecutive calls that reuse its fixed scratch array.

Collected last on purpose, so that a run stopping at its first failure has already run
every other test."""

import dataclasses

import pytest

import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from looped_transformer_kv_gb300 import rq
    from looped_transformer_kv_gb300.workload import Workload


@pytest.mark.parametrize("name,over,ctx", [
    ("pr1_small", {}, [256]),
    ("layer_1p4b", dict(batch=3, n_q_heads=4, n_kv_heads=4), [1000, 64, 3]),
    ("gqa_deep", dict(batch=2, n_q_heads=8, n_kv_heads=2), [700, 129]),
])
def test_noalloc_matches_workspace_entry_point_on_two_calls(name, over, ctx):
    cfg = dataclasses.replace(synth.config_by_name(name), **over)
    w = Workload(cfg, capacity=max(ctx) + 64, ctx_lens=ctx, batch=len(ctx))
    L = cfg.n_loops
    assert rq.decode_workspace_bytes(w.shape, L, w.max_ctx) <= rq.noalloc_scratch_bytes()
    for loop_begin, loop_count in ((0, L), (L - 1, 1), (0, 1)):
        q = w.q[:, :, loop_begin:loop_begin + loop_count].contiguous()
        pend = w.pending[:, :, loop_begin:loop_begin + loop_count].contiguous()
        want = w.out_buffer(loop_count)
        ws = w.workspace(loop_count)
        rq.decode_attention(w.shape, w.cache, q, loop_begin, loop_count, pend, w.ctx_lens,
                            w.max_ctx, want, ws)
        for _ in range(2):                        # the second call reuses the scratch array
            got = torch.full_like(want, float("nan"))
            rq.decode_attention_noalloc(w.shape, w.cache, q, loop_begin, loop_count, pend,
                                        w.ctx_lens, w.max_ctx, got)
            torch.cuda.synchronize()
            assert torch.isfinite(got.float()).all()
            # the same kernels with the same split plan: the same bits
            assert torch.equal(got.view(torch.int16), want.view(torch.int16)), \
                (got.float() - want.float()).abs().max().item()


def test_noalloc_rejects_calls_beyond_its_scratch():
    # a shape whose split-KV scratch needs more than the fixed array: refused, nothing enqueued
    shape = rq.make_shape(4096, 64, 64, 128, 16, 65536, (2,) * 15)
    assert rq.decode_workspace_bytes(shape, 16, 65536) > rq.noalloc_scratch_bytes()
    cache = rq._lib.RqCache()
    cache.data = 256                              # non-null dummies: the call must stop at the
    cache.rot_signs[0] = cache.rot_signs[1] = 16  # size check
    p = rq.ctypes.c_void_p(16)
    status = rq._lib.lib().rq_decode_attention_noalloc(
        rq.ctypes.byref(shape), rq.ctypes.byref(cache), p, 0, 16, None, p, 65536, p, None)
    assert status == 3                            # RQ_ERR_WORKSPACE
