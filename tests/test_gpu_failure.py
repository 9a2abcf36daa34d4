"""Failure paths of the decode kernels, driven without any GPU fault.

- A bounded pipeline wait that runs out: the test hook withholds the copy of each split's first
  tile, so the wait for it can only end by its limit (1 ms here).  Every split with tokens sets
  the workspace error word and returns; its outputs are NaN; the context stays usable and the
  next ordinary call is correct.
- A device-side ctx_len beyond what the call's split grid covers (max_ctx too small, as when a
  captured graph keeps max_ctx fixed while ctx_lens advance): flagged, not silently truncated.
"""

import dataclasses

import pytest

import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from looped_transformer_kv_gb300 import rq
    from looped_transformer_kv_gb300.workload import Workload

LIMIT_NS = 1_000_000


def _err(ws):
    return ws[:1].view(torch.int32).item()


@pytest.mark.parametrize("name,over,ctx,calls", [
    # multi-column blocks: the combine kernel merges the splits
    ("pr1_small", {}, [256], [(0, 4)]),
    ("gqa_deep", dict(batch=2, n_q_heads=8, n_kv_heads=2), [300, 129], [(0, 8), (3, 1)]),
    # single-column blocks (one query head per kv-head, d 128): splits merged in the kernel
    ("layer_1p4b", dict(batch=2, n_q_heads=2, n_kv_heads=2), [450, 300], [(0, 1), (3, 1)]),
])
def test_wait_that_runs_out_flags_the_call_and_leaves_the_context_usable(name, over, ctx, calls):
    cfg = dataclasses.replace(synth.config_by_name(name), **over)
    w = Workload(cfg, capacity=max(ctx) + 64, ctx_lens=ctx, batch=len(ctx))
    for l0, lc in calls:
        q = w.q[:, :, l0:l0 + lc].contiguous()
        pend = w.pending[:, :, l0:l0 + lc].contiguous()
        want, ws0 = w.out_buffer(lc), w.workspace(lc)
        rq.decode_attention(w.shape, w.cache, q, l0, lc, pend, w.ctx_lens, w.max_ctx, want, ws0)
        torch.cuda.synchronize()
        assert _err(ws0) == 0 and torch.isfinite(want.float()).all()
        got, ws = w.out_buffer(lc), w.workspace(lc)
        rq.test_decode_attention_wait_runs_out(w.shape, w.cache, q, l0, lc, pend, w.ctx_lens,
                                               w.max_ctx, got, ws, LIMIT_NS)
        torch.cuda.synchronize()                  # returns: no hang
        assert _err(ws) != 0
        assert torch.isnan(got.float()).all()     # every sequence had cached tokens
        # the context is usable and the same workspace serves an ordinary call again
        again = w.out_buffer(lc)
        rq.decode_attention(w.shape, w.cache, q, l0, lc, pend, w.ctx_lens, w.max_ctx, again, ws)
        torch.cuda.synchronize()
        assert _err(ws) == 0
        assert torch.equal(again.view(torch.int16), want.view(torch.int16))


@pytest.mark.parametrize("lc", [1, 4])
def test_context_beyond_max_ctx_is_flagged(lc):
    cfg = dataclasses.replace(synth.config_by_name("layer_1p4b"), batch=2, n_q_heads=2,
                              n_kv_heads=2)
    w = Workload(cfg, capacity=1024, ctx_lens=[900, 60], batch=2)
    q = w.q[:, :, :lc].contiguous()
    pend = w.pending[:, :, :lc].contiguous()
    small = 64                                    # covers sequence 1, not sequence 0
    ws = w.workspace_for(lc, small)
    out = w.out_buffer(lc)
    rq.decode_attention(w.shape, w.cache, q, 0, lc, pend, w.ctx_lens, small, out, ws)
    torch.cuda.synchronize()
    assert _err(ws) != 0
    assert torch.isnan(out[0].float()).all()      # the truncated sequence is not returned
