"""Serving step under a CUDA graph: per-loop decode of every loop, deferred-write encode of
the current token into slot ctx_len, ctx_len advanced on the device -- captured once and
replayed token after token.  N replays must leave the cache and ctx_lens exactly as N eager
steps do, and produce the same outputs bit for bit (the eager calls are checked against the
fp64 oracle by test_gpu_parity.py)."""

import dataclasses

import pytest

import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from looped_transformer_kv_gb300.workload import Workload


def _arrays(cache):
    out = list(cache.ref_codes) + list(cache.ref_meta)
    for kv in range(2):
        out += cache.res_codes[kv] + cache.res_meta[kv] + cache.alpha[kv]
    return out


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
    for a, b in zip(_arrays(w_graph.cache), _arrays(w_eager.cache)):
        assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))
    for a, b in zip(outs["g"], outs["e"]):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert wss["g"][:1].view(torch.int32).item() == 0
