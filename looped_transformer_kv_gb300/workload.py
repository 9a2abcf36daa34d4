"""Device-resident synthetic workloads: packed cache, BF16 cache, queries, pending tokens.

Inputs come from the seeded generator (the `synth` package's recipe, run on the GPU by
librq's synthetic-input kernel), then the packed cache is built by librq's encode
(bulk deferred write of positions 0..capacity-1, in token chunks so that no full BF16 copy
of the cache is needed).
"""

import numpy as np
import torch

import synth

from . import rq


class Workload:
    def __init__(self, cfg, layer=0, capacity=None, ctx_lens=None, build_rq=True,
                 build_bf16=False, chunk_tokens=2048, device="cuda", batch=None, alpha_mode=0):
        self.cfg = cfg
        self.layer = layer
        self.alpha_mode = alpha_mode     # 0: the method; 1 / 2: a fixed at 1 / 0 (ablations)
        self.device = device
        B = cfg.batch if batch is None else batch
        H, Hq, d, L = cfg.n_kv_heads, cfg.n_q_heads, cfg.head_dim, cfg.n_loops
        cap = cfg.ctx if capacity is None else capacity
        cap = max(64, -(-cap // 64) * 64)                # whole 64-token tiles
        self.B, self.H, self.Hq, self.d, self.L, self.cap = B, H, Hq, d, L, cap
        if ctx_lens is None:
            ctx_lens = [min(cfg.ctx, cap)] * B
        self.ctx_list = [int(c) for c in ctx_lens]
        assert len(self.ctx_list) == B and all(0 <= c <= cap for c in self.ctx_list)
        self.max_ctx = max(self.ctx_list) if B else 0
        self.ctx_lens = torch.tensor(self.ctx_list, dtype=torch.int32, device=device)
        self.shape = rq.make_shape(B, Hq, H, d, L, cap, cfg.res_bits[: L - 1])
        signs = synth.rotation_signs(cfg, layer)                      # [H][2][d]
        self.signs_np = signs
        self.outliers = torch.from_numpy(synth.outlier_table(cfg, layer)).to(device)
        self.params = rq.synth_params(cfg.seed, layer, d, H, cfg.dist, cfg.sigma,
                                      cfg.outlier_mult, self.outliers if cfg.n_outliers else None)
        self.cache = None
        if build_rq:
            self.cache = rq.PackedCache(self.shape, torch.from_numpy(signs.transpose(1, 0, 2).copy()),
                                        device=device)
            self._build_rq(chunk_tokens)
        self.k = self.v = None
        if build_bf16:
            self._build_bf16()
        # queries [B][Hq][L][d] and the pending (current) token at position ctx_len[b]
        self.q = torch.empty(B, Hq, L, d, dtype=torch.bfloat16, device=device)
        rq.synth_queries(self.params, self.q, Hq, 0, B, 0, L)
        self.pending = torch.empty(B, 2, L, H, d, dtype=torch.bfloat16, device=device)
        st = self.pending.stride()
        for b in range(B):
            rq.synth_states(self.params, self.pending[b], (0, 0, st[1], st[2], st[3]),
                            b, 1, self.ctx_list[b], 1, 0, L)
        self.q_loop = [self.q[:, :, l:l + 1].contiguous() for l in range(L)]
        self.pending_loop = [self.pending[:, :, l:l + 1].contiguous() for l in range(L)]

    # ------------------------------------------------------------------ builders
    def _build_rq(self, chunk_tokens):
        B, H, d, L, cap = self.B, self.H, self.d, self.L, self.cap
        bmax = max(1, min(B, (1 << 28) // max(1, chunk_tokens * 2 * L * H * d)))
        buf = torch.empty(bmax, chunk_tokens, 2, L, H, d, dtype=torch.bfloat16, device=self.device)
        st = buf.stride()
        for b0 in range(0, B, bmax):
            nb = min(bmax, B - b0)
            for t0 in range(0, cap, chunk_tokens):
                nt = min(chunk_tokens, cap - t0)
                rq.synth_states(self.params, buf, st[:5], b0, nb, t0, nt, 0, L)
                view = buf[:nb, :nt]
                sub = rq.make_shape(nb, self.Hq, H, d, L, cap, self.cfg.res_bits[: L - 1])
                sub_cache = self._sub_cache(b0, nb)
                if self.alpha_mode:
                    rq.ablation_encode_append(sub, sub_cache, view, self.alpha_mode, pos_begin=t0)
                else:
                    rq.encode_append(sub, sub_cache, view, pos_begin=t0)
        del buf

    def _sub_cache(self, b0, nb):
        """A view of the cache restricted to sequences [b0, b0+nb) (a pointer offset: the
        records of a sequence are contiguous)."""
        c = rq._lib.RqCache()
        full = self.cache
        c.data = full.data.data_ptr() + b0 * self.H * (self.cap // rq.PAGE) * full.rec
        for kv in range(2):
            c.rot_signs[kv] = full.rot_signs[kv].data_ptr()

        class _V:
            pass

        v = _V()
        v.struct = c
        return v

    def _build_bf16(self):
        B, H, d, L, cap = self.B, self.H, self.d, self.L, self.cap
        kv = torch.empty(2, B, H, L, cap, d, dtype=torch.bfloat16, device=self.device)
        s = kv.stride()                      # (kv, b, h, l, t, i)
        rq.synth_states(self.params, kv, (s[1], s[4], s[0], s[3], s[2]), 0, B, 0, cap, 0, L)
        self.kv_bf16 = kv
        self.k, self.v = kv[0], kv[1]

    # ------------------------------------------------------------------ calls
    def workspace(self, loop_count):
        n = rq.decode_workspace_bytes(self.shape, loop_count, self.max_ctx)
        return torch.empty(max(n, 16) // 4 + 4, dtype=torch.float32, device=self.device)

    def decode(self, loop_begin, loop_count, out, ws, pending=True, stream=None):
        q = self.q if loop_count == self.L else (
            self.q_loop[loop_begin] if loop_count == 1 else
            self.q[:, :, loop_begin:loop_begin + loop_count].contiguous())
        pend = None
        if pending:
            pend = self.pending if loop_count == self.L else (
                self.pending_loop[loop_begin] if loop_count == 1 else
                self.pending[:, :, loop_begin:loop_begin + loop_count].contiguous())
        rq.decode_attention(self.shape, self.cache, q, loop_begin, loop_count, pend,
                            self.ctx_lens, self.max_ctx, out, ws, stream)

    def decode_ablation(self, loop, out, ws, pending=True, stream=None):
        """Per-loop decode of residual loop `loop` over this (ablation-encoded) cache."""
        pend = self.pending_loop[loop] if pending else None
        rq.ablation_decode_attention(self.shape, self.cache, self.alpha_mode, self.q_loop[loop],
                                     loop, pend, self.ctx_lens, self.max_ctx, out, ws, stream)

    def decode_bf16(self, loop_begin, loop_count, out, ws, pending=True, stream=None):
        q = self.q if loop_count == self.L else (
            self.q_loop[loop_begin] if loop_count == 1 else
            self.q[:, :, loop_begin:loop_begin + loop_count].contiguous())
        pend = None
        if pending:
            pend = self.pending if loop_count == self.L else (
                self.pending_loop[loop_begin] if loop_count == 1 else
                self.pending[:, :, loop_begin:loop_begin + loop_count].contiguous())
        rq.bf16_decode_attention(self.shape, self.k, self.v, q, loop_begin, loop_count, pend,
                                 self.ctx_lens, self.max_ctx, out, ws, stream)

    def out_buffer(self, loop_count):
        return torch.empty(self.B, self.Hq, loop_count, self.d, dtype=torch.bfloat16,
                           device=self.device)

    # ------------------------------------------------------------------ serving step
    def serving_step(self, ctx_lens, out1, ws1, max_ctx, stream=None):
        """One decode step of the looped model for every sequence, as a server runs it: loop
        l's query attends over loop l's cache with the current token's loop-l state pending,
        for l = 0..L-1 in order; then the token's L states are encoded into slot ctx_len
        (deferred write) and ctx_len advances by one, on the device.  With max_ctx fixed (an
        upper bound), the sequence of calls can be captured once in a CUDA graph and replayed
        token after token."""
        B, L = self.B, self.L
        for l in range(L):
            rq.decode_attention(self.shape, self.cache, self.q_loop[l], l, 1, self.pending_loop[l],
                                ctx_lens, max_ctx, out1[l], ws1, stream)
        kv_new = self.pending.reshape(B, 1, 2, L, self.H, self.d)
        rq.encode_append(self.shape, self.cache, kv_new, positions=ctx_lens, stream=stream)
        rq.advance_ctx(ctx_lens, 1, self.cap, stream)

    def workspace_for(self, loop_count, max_ctx):
        n = rq.decode_workspace_bytes(self.shape, loop_count, max_ctx)
        return torch.empty(max(n, 16) // 4 + 4, dtype=torch.float32, device=self.device)

    # ------------------------------------------------------------------ paged twin
    def paged_twin(self, spare_pages=0, seed=0, chunk_tokens=2048):
        """The same tokens in a paged cache (64-token pages scattered at random over a pool of
        B * capacity / 64 + spare_pages pages).  Returns (cache, paging, block_table)."""
        B, H, d, L, cap = self.B, self.H, self.d, self.L, self.cap
        max_pages = cap // rq.PAGE
        n_pages = B * max_pages + spare_pages
        rng = np.random.default_rng(seed)
        table = rng.permutation(n_pages)[: B * max_pages].reshape(B, max_pages).astype(np.int32)
        bt = torch.from_numpy(table).to(self.device)
        signs = torch.from_numpy(self.signs_np.transpose(1, 0, 2).copy())
        pc = rq.PackedCache(self.shape, signs, device=self.device, n_pages=n_pages)
        paging = rq.make_paging(bt, n_pages)
        bmax = max(1, min(B, (1 << 28) // max(1, chunk_tokens * 2 * L * H * d)))
        buf = torch.empty(bmax, chunk_tokens, 2, L, H, d, dtype=torch.bfloat16, device=self.device)
        st = buf.stride()
        for b0 in range(0, B, bmax):
            nb = min(bmax, B - b0)
            sub = rq.make_shape(nb, self.Hq, H, d, L, cap, self.cfg.res_bits[: L - 1])
            sub_paging = rq.make_paging(bt[b0:b0 + nb], n_pages)
            for t0 in range(0, cap, chunk_tokens):
                nt = min(chunk_tokens, cap - t0)
                rq.synth_states(self.params, buf, st[:5], b0, nb, t0, nt, 0, L)
                rq.paged_encode_append(sub, pc, sub_paging, buf[:nb, :nt], pos_begin=t0)
        del buf
        return pc, paging, bt

    def decode_paged(self, cache, paging, loop_begin, loop_count, out, ws, pending=True,
                     stream=None):
        q = self.q if loop_count == self.L else (
            self.q_loop[loop_begin] if loop_count == 1 else
            self.q[:, :, loop_begin:loop_begin + loop_count].contiguous())
        pend = None
        if pending:
            pend = self.pending if loop_count == self.L else (
                self.pending_loop[loop_begin] if loop_count == 1 else
                self.pending[:, :, loop_begin:loop_begin + loop_count].contiguous())
        rq.paged_decode_attention(self.shape, cache, paging, q, loop_begin, loop_count, pend,
                                  self.ctx_lens, self.max_ctx, out, ws, stream)

    # ------------------------------------------------------------------ readback
    def packed_slice_paged(self, pc, table, b, h, ntok):
        """packed_slice of a paged cache `pc` whose block table is `table` (host [B][pages])."""
        ntok += ntok % 2
        npg = -(-ntok // rq.PAGE)
        idx = torch.as_tensor(np.asarray(table[b][:npg], dtype=np.int64), device=pc.data.device)
        return slice_from_records(pc, pc.records()[idx, h], ntok)

    def packed_slice(self, b, h, ntok):
        """Host copies of the packed arrays of (sequence b, kv-head h), tokens [0, ntok)."""
        ntok += ntok % 2
        npg = -(-ntok // rq.PAGE)
        return slice_from_records(self.cache, self.cache.records()[b, h, :npg], ntok)


def slice_from_records(pc, recs, ntok):
    """The packed arrays of one (sequence, kv-head) of cache `pc` from its records [n][rec]
    (uint8, on the device), tokens [0, ntok): each kind of row concatenated over the records
    ({("ref_codes", kv): uint8 [ntok][row], ("ref_meta", kv): [ntok][ng][2], per loop l
    ("res_codes", kv, l), ("res_meta", kv, l), ("alpha", kv, l): [ntok]}; fp16 as float32)."""
    d, L = pc.shape.head_dim, pc.shape.n_loops
    ng = d // rq.GROUP
    out = {}

    def rows(kind, kv, loop=None, dtype=None):
        off, rb = pc.section(kind, kv, loop)
        a = recs[:, off:off + rq.PAGE * rb].reshape(-1, rb)[:ntok]
        if dtype is None:
            return a.cpu().numpy()
        return a.contiguous().view(dtype).float().cpu().numpy()

    for kv in range(2):
        out[("ref_codes", kv)] = rows("codes", kv)
        out[("ref_meta", kv)] = rows("meta", kv, None, torch.float16).reshape(ntok, ng, 2)
        for l in range(L - 1):
            out[("res_codes", kv, l)] = rows("codes", kv, l)
            out[("res_meta", kv, l)] = rows("meta", kv, l, torch.float16).reshape(ntok, ng, 2)
            out[("alpha", kv, l)] = rows("alpha", kv, l, torch.float16).reshape(ntok)
    return out


def np_bf16(t):
    """bf16 torch tensor -> fp64 numpy."""
    return t.float().cpu().numpy().astype(np.float64)


def budget_batches(cfg, budget_bytes, capacity):
    """Fixed KV-memory budget for one layer: the largest batch whose packed cache fits
    `budget_bytes`, and the largest whose BF16 cache ([B][Hkv][L][capacity][d], K and V) does.
    Returns (rq_batch, bf16_batch, rq_bytes_per_sequence, bf16_bytes_per_sequence)."""
    L, H, d = cfg.n_loops, cfg.n_kv_heads, cfg.head_dim
    rq_seq = rq.cache_bytes(rq.make_shape(1, cfg.n_q_heads, H, d, L, capacity,
                                          cfg.res_bits[: L - 1]))
    bf_seq = 2 * H * L * capacity * d * 2
    return int(budget_bytes // rq_seq), int(budget_bytes // bf_seq), int(rq_seq), int(bf_seq)
