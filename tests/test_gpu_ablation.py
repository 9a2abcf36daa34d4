"""Ablation rows on the GPU: caches encoded with a fixed at 1 or 0 (rq_ablation_encode_append)
and their per-loop decode kernels (rq_ablation_decode_attention: a = 1 without reading the a
stream; a = 0 without reading the reference), against the fp64 oracle's steps with the same
change, and against the method's decode kernel run over the same cache (which reads the fixed
a and, for a = 0, a reference whose contribution is exactly zero: the same bits)."""

import dataclasses
import functools

import pytest

import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from looped_transformer_kv_gb300.workload import Workload

from ablation import encode_fixed_alpha  # noqa: E402
from rq_parity import check_slice  # noqa: E402


@pytest.mark.parametrize("mode", [1, 2])
@pytest.mark.parametrize("name,over,ctx", [
    ("layer_1p4b", dict(batch=2, n_q_heads=2, n_kv_heads=2), [300, 65]),
    ("mixed_24l", dict(batch=2, n_q_heads=2, n_kv_heads=2), [129, 0]),   # 4-bit loop 0
])
def test_ablation_decode_matches_oracle_and_method_kernel(mode, name, over, ctx):
    cfg = dataclasses.replace(synth.config_by_name(name), **over)
    w = Workload(cfg, capacity=max(ctx) + 64, ctx_lens=ctx, batch=len(ctx), alpha_mode=mode)
    L = cfg.n_loops
    calls, outs = [], []
    for l in range(L - 1):
        o, ws = w.out_buffer(1), w.workspace(1)
        w.decode_ablation(l, o, ws)
        ref_o, ref_ws = w.out_buffer(1), w.workspace(1)
        w.decode(l, 1, ref_o, ref_ws)            # the method's kernel over the same cache
        torch.cuda.synchronize()
        assert ws[:1].view(torch.int32).item() == 0
        assert torch.equal(o.view(torch.int16), ref_o.view(torch.int16)), l
        calls.append((l, 1))
        outs.append(o)
    enc = functools.partial(encode_fixed_alpha, a_value=1.0 if mode == 1 else 0.0)
    for b in range(w.B):
        for h in range(w.H):
            check_slice(w, b, h, calls, outs, encode=enc)
