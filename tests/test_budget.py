"""Fixed KV-memory budget experiment: the batch each cache format fits in a budget (CPU), and a
decode at the packed cache's budget batch checked against the fp64 oracle (GPU)."""

import dataclasses

import pytest

import oracle as O
import synth


def _cfg():
    return dataclasses.replace(synth.config_by_name("layer_1p4b"), batch=1, n_q_heads=2,
                               n_kv_heads=2, ctx=256)


def test_budget_batches_are_the_largest_that_fit():
    from looped_transformer_kv_gb300 import build
    build.build()
    from looped_transformer_kv_gb300.workload import budget_batches
    cfg = _cfg()
    cap, budget = 320, 2 << 20
    b_rq, b_bf, rq_seq, bf_seq = budget_batches(cfg, budget, cap)
    assert rq_seq == O.cache_bytes(cfg.head_dim, cfg.n_loops, cfg.res_bits, cap, cfg.n_kv_heads)
    assert bf_seq == 2 * cfg.n_kv_heads * cfg.n_loops * cap * cfg.head_dim * 2
    assert b_rq * rq_seq <= budget < (b_rq + 1) * rq_seq
    assert b_bf * bf_seq <= budget < (b_bf + 1) * bf_seq
    assert b_rq > 4 * b_bf                          # 2-bit residuals: more than 4x the batch


@pytest.mark.gpu
def test_decode_at_the_budget_batch_matches_the_oracle():
    torch = pytest.importorskip("torch")
    from looped_transformer_kv_gb300.workload import Workload, budget_batches
    from rq_parity import check_slice
    cfg = _cfg()
    cap, budget = 320, 2 << 20
    b_rq, _, rq_seq, _ = budget_batches(cfg, budget, cap)
    w = Workload(cfg, capacity=cap, batch=b_rq)
    assert w.cache.nbytes() == b_rq * rq_seq <= budget
    L = cfg.n_loops
    out, ws = w.out_buffer(L), w.workspace(L)
    w.decode(0, L, out, ws)
    torch.cuda.synchronize()
    assert ws[:1].view(torch.int32).item() == 0
    check_slice(w, b_rq - 1, cfg.n_kv_heads - 1, [(0, L)], [out])
