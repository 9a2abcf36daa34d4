"""Serving step under a CUDA graph: per-loop decode of every loop, deferred-write encode of
the current token into slot ctx_len, ctx_len advanced on the device -- captured once and
replayed token after token.  N replays must leave the cache and ctx_lens exactly as N eager
steps do, and produce the same outputs bit for bit.  The replayed run is also checked against
the fp64 oracle on its own: the grown cache (ctx original tokens, then N appended copies of the
current token) is re-encoded by the oracle and compared code for code, and the last step's
per-loop outputs (ctx + N - 1 cached tokens plus the current token) are recomputed."""

import dataclasses

import numpy as np
import pytest

import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from looped_transformer_kv_gb300.workload import Workload

from rq_parity import check_slice  # noqa: E402


@pytest.mark.parametrize("name,over,ctx", [
    ("pr1_small", {}, [100]),
    ("layer_1p4b", dict(batch=2, n_q_heads=2, n_kv_heads=2), [130, 0]),
    ("mixed_24l", dict(batch=2, n_q_heads=4, n_kv_heads=2), [61, 64]),
])
def test_graph_replayed_serving_steps_match_eager_steps(name, over, ctx):
    cfg = dataclasses.replace(synth.config_by_name(name), **over)
    cap, steps = 256, 4
    w_graph = Workload(cfg, capacity=cap, ctx_lens=ctx, batch=len(ctx))
    w_eager = Workload(cfg, capacity=cap, ctx_lens=ctx, batch=len(ctx))
    L = cfg.n_loops
    outs = {k: [w.out_buffer(1) for _ in range(L)] for k, w in (("g", w_graph), ("e", w_eager))}
    wss = {k: w.workspace_for(1, cap) for k, w in (("g", w_graph), ("e", w_eager))}
    ctx_g = w_graph.ctx_lens.clone()
    ctx_e = w_eager.ctx_lens.clone()
    # eager steps
    for _ in range(steps):
        w_eager.serving_step(ctx_e, outs["e"], wss["e"], cap)
    torch.cuda.synchronize()
    # one capture, then replays (the capture itself runs nothing)
    side = torch.cuda.Stream()
    with torch.cuda.stream(side):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=side):
            w_graph.serving_step(ctx_g, outs["g"], wss["g"], cap)
    torch.cuda.synchronize()
    for _ in range(steps):
        g.replay()
    torch.cuda.synchronize()
    assert ctx_g.tolist() == ctx_e.tolist() == [min(c + steps, cap) for c in ctx]
    assert torch.equal(w_graph.cache.data, w_eager.cache.data)
    for a, b in zip(outs["g"], outs["e"]):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert wss["g"][:1].view(torch.int32).item() == 0
    # the replayed run against the oracle: each sequence's cache grew by `steps` copies of its
    # current token (the deferred writes), and the last step attended over all but the last
    calls = [(l, 1) for l in range(L)]
    for b, c0 in enumerate(ctx):
        n = c0 + steps
        for h in sorted({0, w_graph.H - 1}):
            x = synth.gen_states(cfg, 0, [b], np.arange(n + n % 2), heads=[h])[0, :, :, :, 0, :]
            pend = synth.gen_states(cfg, 0, [b], [c0], heads=[h])[0, 0, :, :, 0, :]
            x[c0:n] = pend
            check_slice(w_graph, b, h, calls, outs["g"], states=x, ctx=n - 1, pending_state=pend)
