"""Paged cache (block table of 64-token pages) against the contiguous cache, on the GPU.

The same seeded states are encoded into a contiguous cache and into a paged cache whose
block table scatters every sequence's pages over a larger pool in random order.  Every
page of the paged arrays must equal the matching 64-token rows of the contiguous arrays
byte for byte, and the paged decode must return the contiguous decode's outputs bit for bit
(the contiguous path itself is checked against the fp64 oracle by test_gpu_parity.py).
"""

import dataclasses

import numpy as np
import pytest

import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import looped_transformer_kv_gb300 as rqm
    from looped_transformer_kv_gb300.workload import Workload

from rq_parity import check_slice  # noqa: E402


def _cfg(name, **kw):
    return dataclasses.replace(synth.config_by_name(name), **kw)


CASES = [
    ("pr1_small", {}, [256]),
    ("layer_1p4b", dict(batch=3, n_q_heads=2, n_kv_heads=2), [257, 64, 1]),
    ("gqa_deep", dict(batch=2, n_q_heads=8, n_kv_heads=2), [300, 129]),
    ("mixed_24l", dict(batch=2, n_q_heads=2, n_kv_heads=2), [191, 0]),
]


def _paged_twin(w, spare_pages, seed):
    """A paged cache holding the same tokens as workload w, pages scattered at random."""
    pc, paging, bt = w.paged_twin(spare_pages=spare_pages, seed=seed)
    return pc, paging, bt, bt.cpu().numpy()


@pytest.mark.parametrize("case", range(len(CASES)))
def test_paged_cache_matches_contiguous(case):
    name, over, ctx = CASES[case]
    cfg = _cfg(name, **over)
    cap = -(-(max(ctx) + 2) // 64) * 64
    w = Workload(cfg, capacity=cap, ctx_lens=ctx, batch=len(ctx))
    pc, paging, bt, table = _paged_twin(w, spare_pages=5, seed=case)
    torch.cuda.synchronize()
    # every page's records byte for byte
    c = w.cache.records()                                    # [B][H][pages][rec]
    p = pc.records()                                         # [n_pages][H][rec]
    for b in range(w.B):
        got = p[torch.from_numpy(table[b]).long().cuda()]    # [pages][H][rec]
        want = c[b].permute(1, 0, 2)                          # [pages][H][rec]
        assert torch.equal(got, want), b
    # decode: all loops at once, each loop alone, a middle range
    calls = [(0, cfg.n_loops)] + [(l, 1) for l in range(cfg.n_loops)]
    if cfg.n_loops > 2:
        calls.append((1, 2))
    paged_outs = []
    for l0, lc in calls:
        o1, o2 = w.out_buffer(lc), w.out_buffer(lc)
        ws1, ws2 = w.workspace(lc), w.workspace(lc)
        w.decode(l0, lc, o1, ws1)
        q = w.q[:, :, l0:l0 + lc].contiguous()
        pend = w.pending[:, :, l0:l0 + lc].contiguous()
        rqm.rq.paged_decode_attention(w.shape, pc, paging, q, l0, lc, pend, w.ctx_lens,
                                      w.max_ctx, o2, ws2)
        torch.cuda.synchronize()
        assert ws2[:1].view(torch.int32).item() == 0
        assert torch.equal(o1.view(torch.int16), o2.view(torch.int16)), (l0, lc)
        paged_outs.append(o2)
    # the paged cache's pages and the paged outputs against the oracle, every sequence
    for b in range(w.B):
        for h in sorted({0, w.H - 1}):
            check_slice(w, b, h, calls, paged_outs, cache=(pc, table))


def test_paged_table_entry_out_of_range_is_flagged_not_read():
    cfg = _cfg("pr1_small")
    w = Workload(cfg, capacity=256, ctx_lens=[200], batch=1)
    pc, paging, bt, table = _paged_twin(w, spare_pages=0, seed=9)
    bad = bt.clone()
    bad[0, 1] = pc.n_pages + 7                    # page 1 of sequence 0: out of range
    bad_paging = rqm.rq.make_paging(bad, pc.n_pages)
    L = cfg.n_loops
    o, ws = w.out_buffer(L), w.workspace(L)
    rqm.rq.paged_decode_attention(w.shape, pc, bad_paging, w.q, 0, L, w.pending, w.ctx_lens,
                                  w.max_ctx, o, ws)
    torch.cuda.synchronize()
    assert ws[:1].view(torch.int32).item() != 0
    assert torch.isnan(o.float()).all()
    # encode: the token whose page is out of range is skipped, the others are written
    before = pc.records().clone()
    kv = torch.zeros(1, 2, 2, L, w.H, w.d, dtype=torch.bfloat16, device="cuda")
    pos = torch.tensor([[70, 10]], dtype=torch.int32, device="cuda")   # page 1 (bad), page 0
    rqm.rq.paged_encode_append(w.shape, pc, bad_paging, kv, positions=pos)
    torch.cuda.synchronize()
    after = pc.records()
    assert not torch.equal(before, after)          # token 10 (page 0) was written
    p1 = int(table[0, 1])
    assert torch.equal(before[p1], after[p1])      # page 1's records untouched


def test_bad_table_entry_in_single_column_calls_gives_nan():
    # one query head per kv-head and head dim 128: the per-loop calls run the single-column
    # variants, which merge their splits in the split kernel; the error word is set and every
    # output of the sequence whose split met the bad entry is NaN (the other sequence's units
    # may have merged before the flag)
    cfg = _cfg("layer_1p4b", batch=2, n_q_heads=2, n_kv_heads=2)
    w = Workload(cfg, capacity=512, ctx_lens=[450, 300], batch=2)
    pc, paging, bt, table = _paged_twin(w, spare_pages=0, seed=11)
    good = w.out_buffer(1), w.workspace(1)
    q = w.q[:, :, 0:1].contiguous()
    pend = w.pending[:, :, 0:1].contiguous()
    rqm.rq.paged_decode_attention(w.shape, pc, paging, q, 0, 1, pend, w.ctx_lens, w.max_ctx,
                                  good[0], good[1])
    torch.cuda.synchronize()
    assert good[1][:1].view(torch.int32).item() == 0
    assert torch.isfinite(good[0].float()).all()
    bad = bt.clone()
    bad[1, 2] = -3                                  # sequence 1, page 2: out of range
    o, ws = w.out_buffer(1), w.workspace(1)
    rqm.rq.paged_decode_attention(w.shape, pc, rqm.rq.make_paging(bad, pc.n_pages), q, 0, 1, pend,
                                  w.ctx_lens, w.max_ctx, o, ws)
    torch.cuda.synchronize()
    assert ws[:1].view(torch.int32).item() != 0
    assert torch.isnan(o[1].float()).all()
