#!/usr/bin/env python
"""Decode-attention benchmark of librq on one GB300 (one JSON line on stdout).

A step is one decode step of one layer of a looped model on the workload's batch: fused
decode attention of every loop over the packed cache (all loops' queries in one call, the
reference tile read once) plus the deferred write of the current token (encode + append of
its L loop states).  Metric: KV tokens/s = batch * ctx * loops * layers / step time.

python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

With --gpus N > 1 (launched by torch.distributed.run) every rank runs the whole workload on
its own GPU (independent sequences: weak scaling, no collective on the data path); times
are max-reduced over ranks.  --impl reference times the fp64 CPU oracle on host cores.
"""

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode-attn KV tokens/s at 1 GB300, HBM GB/s vs peak, vs in-build BF16 kernel"

# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) of one all-loops decode launch
# of the split kernel, from one ncu capture (profiles/), keyed by the kernel sources they
# were taken on; any change to those sources makes the figure stale (reported as null).
KERNEL_SOURCES = ("looped_transformer_kv_gb300/csrc/rq_decode_mma.cu",
                  "looped_transformer_kv_gb300/csrc/rq_decode_mma.cuh",
                  "looped_transformer_kv_gb300/csrc/rq_ptx.cuh",
                  "looped_transformer_kv_gb300/csrc/rq_common.cuh",
                  "looped_transformer_kv_gb300/csrc/rq_kernels.h")
TRAFFIC = {
    ("7a5789489900c373", "layer_1p4b"): 483010304 + 11158272,  # profiles/rq_mma_kernel_layer_1p4b.md
}


def _kernel_hash():
    import hashlib
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def _traffic(workload):
    t = TRAFFIC.get((_kernel_hash(), workload))
    return t


def reduce_step_ms(ms, world):
    """Max of the per-rank step times over all ranks (every rank gets the max)."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


# ---------------------------------------------------------------------------- oracle arm

ORACLE_SNIPPET = r"""
import json, sys, time
import numpy as np
sys.path.insert(0, %(root)r)
import oracle as O, synth
cfg = synth.config_by_name(%(name)r)
heads = %(heads)r
slices = []
for h in heads:
    x = synth.gen_states(cfg, 0, [0], np.arange(cfg.ctx + 1), heads=[h])[0, :, :, :, 0, :].astype(np.float64)
    s = synth.rotation_signs(cfg, 0)[h].astype(np.float64)
    rb = cfg.res_bits[: cfg.n_loops - 1]
    ek = O.encode(x[:cfg.ctx, 0], s[0], rb)
    ev = O.encode(x[:cfg.ctx, 1], s[1], rb)
    q = synth.gen_queries(cfg, 0, [0])[0].astype(np.float64)
    g = cfg.n_q_heads // cfg.n_kv_heads
    slices.append((ek, ev, s, q[h * g:(h + 1) * g], x[cfg.ctx]))
def one_pass():
    for ek, ev, s, q, pend in slices:
        for l in range(cfg.n_loops):
            O.decode_rotated(q[:, l], ek, ev, s[0], s[1], l, pend[0, l], pend[1, l])
tok = len(slices) * cfg.ctx * cfg.n_loops
times = []
for i in range(%(warmup)d):
    one_pass()
t_all = time.perf_counter()
reps = 0
while True:
    t0 = time.perf_counter(); one_pass(); times.append(time.perf_counter() - t0); reps += 1
    if reps >= %(min_reps)d and time.perf_counter() - t_all >= %(min_s)f:
        break
print(json.dumps({"times": times, "tokens_per_pass": tok}))
"""


def run_oracle(name, heads, warmup, min_reps, min_s):
    env = dict(os.environ)
    n = os.cpu_count() or 1
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        env[k] = str(n)
    code = ORACLE_SNIPPET % dict(root=ROOT, name=name, heads=list(heads), warmup=warmup,
                                 min_reps=min_reps, min_s=min_s)
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env)
    if r.returncode != 0:
        raise RuntimeError("oracle run failed: " + r.stderr[-2000:])
    d = json.loads(r.stdout.strip().splitlines()[-1])
    return d["times"], d["tokens_per_pass"], n


def reference_arm(args, cfg):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    heads = [0]
    times, tok, cores = run_oracle(cfg.name, heads, args.warmup, args.steps, 0.0)
    times = times[: args.steps]
    t = sum(times)
    value = tok * len(times) / t
    sample = ("sequence 0, kv-head 0: fp64 oracle decode (rotated form) of all %d loops over "
              "ctx %d per step" % (cfg.n_loops, cfg.ctx))
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "KV tokens/s",
            "n_gpus": args.gpus, "steps": len(times), "warmup": args.warmup,
            "ms_per_step": 1e3 * t / len(times), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": _workload_desc(cfg), "sample": sample},
            "cpu_baseline": {"value": value, "unit": "KV tokens/s", "cores": cores,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "KV tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------- GPU arm

def _workload_desc(cfg):
    return ("%s: B %d, Hq %d / Hkv %d, d %d, %d loops (INT4 ref, residual bits %s), ctx %d, "
            "group 32, layers %d" % (cfg.name, cfg.batch, cfg.n_q_heads, cfg.n_kv_heads,
                                     cfg.head_dim, cfg.n_loops,
                                     "/".join(str(b) for b in cfg.res_bits), cfg.ctx, cfg.layers))


class Clocks:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.p = None
        try:
            self.p = subprocess.Popen(["nvidia-smi", "-i", str(index), "--query-gpu=" + self.FIELDS,
                                       "--format=csv,noheader,nounits", "-lms", "200"],
                                      stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.p = None

    def stop(self):
        if self.p is None:
            return None
        self.p.terminate()
        try:
            out, _ = self.p.communicate(timeout=5)
        except Exception:
            self.p.kill()
            out, _ = self.p.communicate()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


def gpu_arm(args, cfg):
    import torch
    import torch.distributed as dist

    import looped_transformer_kv_gb300 as rqm
    from looped_transformer_kv_gb300.workload import Workload

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("gloo")
    torch.cuda.set_device(local)

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        # the oracle runs in a fresh process before this one touches the GPU
        times, tok, cores = run_oracle(cfg.name, list(range(min(4, cfg.n_kv_heads))), 1, 1,
                                       args.cpu_seconds)
        cpu = {"value": tok * len(times) / sum(times), "unit": "KV tokens/s", "cores": cores,
               "kind": "oracle",
               "sample": "sequence 0, kv-heads 0..%d (ctx %d, all %d loops), fp64 oracle decode "
                         "(rotated form) repeated %d times, %.1f s" %
                         (min(4, cfg.n_kv_heads) - 1, cfg.ctx, cfg.n_loops, len(times),
                          sum(times))}

    # spare slots past ctx: the deferred write of the current token lands in slot ctx,
    # which the step's attention (ctx_lens = ctx) does not read, so every step is the same.
    # Every layer of the model gets its own packed cache (the BF16 cache of one layer is
    # built for the comparison kernel: the same shapes for every layer).
    layers = [Workload(cfg, layer=l, capacity=cfg.ctx + 2, build_bf16=(l == 0 and not args.no_bf16))
              for l in range(cfg.layers)]
    w = layers[0]
    NL = len(layers)
    L, B, ctx = cfg.n_loops, w.B, cfg.ctx
    stream = torch.cuda.current_stream()
    out = w.out_buffer(L)
    ws = w.workspace(L)
    ws1 = w.workspace(1)
    out1 = [w.out_buffer(1) for _ in range(L)]
    # deferred write of the current token: its L states, appended at slot ctx
    new_kv = w.pending.reshape(B, 1, 2, L, w.H, w.d)
    pos_new = torch.full((B, 1), ctx, dtype=torch.int32, device="cuda")

    outs = [out] + [lw.out_buffer(L) for lw in layers[1:]]

    def step():
        for lw, o in zip(layers, outs):
            lw.decode(0, L, o, ws)
            rqm.encode_append(lw.shape, lw.cache, lw.pending.reshape(B, 1, 2, L, w.H, w.d),
                              positions=pos_new)

    g = w.Hq // w.H
    # split-kernel blocks, the combine (single-column calls combine inside the split kernel),
    # the encode
    combine = 0 if (g * L == 1 and w.d == 128) else 1
    launches_per_step = NL * (math.ceil(g * L / 8) + combine + 1)

    def graph_of(fn):
        """Capture fn (a sequence of library calls on the current stream) in a CUDA graph."""
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            fn()
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr):
            fn()
        torch.cuda.synchronize()
        return gr

    def timeit(gr, iters):
        """Per-replay device times (ms) of a captured graph, CUDA events on this stream."""
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(iters + 1)]
        torch.cuda.synchronize()
        ev[0].record(stream)
        for i in range(iters):
            gr.replay()
            ev[i + 1].record(stream)
        torch.cuda.synchronize()
        return [ev[i].elapsed_time(ev[i + 1]) for i in range(iters)]

    g_step = graph_of(step)
    # ---- warm-up, then the timed steps (barrier + synchronize on both sides) ----
    for _ in range(args.warmup):
        g_step.replay()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clocks = Clocks(local)
    time.sleep(0.3)
    torch.cuda.synchronize()
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for _ in range(args.steps):
        g_step.replay()
    stop.record(stream)
    torch.cuda.synchronize()
    ms = start.elapsed_time(stop) / args.steps
    ms = reduce_step_ms(ms, world)
    if world > 1:
        dist.barrier()

    # ---- per-call timings (graph replays, same stream, CUDA events) ----
    iters = max(args.steps, 20)
    t_dec = timeit(graph_of(lambda: w.decode(0, L, out, ws)), iters)
    t_enc = timeit(graph_of(lambda: rqm.encode_append(w.shape, w.cache, new_kv, positions=pos_new)),
                   iters)

    def perloop():
        for l in range(L):
            w.decode(l, 1, out1[l], ws1)

    t_per = timeit(graph_of(perloop), iters)
    t_bf_multi = t_bf_per = None
    if not args.no_bf16:
        t_bf_multi = timeit(graph_of(lambda: w.decode_bf16(0, L, out, ws)), iters)

        def bf_per():
            for l in range(L):
                w.decode_bf16(l, 1, out1[l], ws1)

        t_bf_per = timeit(graph_of(bf_per), iters)
    # the same tokens in a paged cache (64-token pages scattered over a pool with spare pages)
    t_pg_multi = t_pg_per = None
    if not args.no_paged:
        pc, paging, bt = w.paged_twin(spare_pages=64, seed=1)
        t_pg_multi = timeit(graph_of(lambda: w.decode_paged(pc, paging, 0, L, out, ws)), iters)

        def pg_per():
            for l in range(L):
                w.decode_paged(pc, paging, l, 1, out1[l], ws1)

        t_pg_per = timeit(graph_of(pg_per), iters)
        del pc, paging, bt
        torch.cuda.empty_cache()
    # serving step: the L per-loop decode calls, the deferred write of the token into slot
    # ctx_len and the advance of ctx_len, captured once and replayed token after token (the
    # spare capacity past ctx takes the appended tokens)
    ctx_srv = w.ctx_lens.clone()
    ws_srv = w.workspace_for(1, w.cap)
    t_srv = timeit(graph_of(lambda: w.serving_step(ctx_srv, out1, ws_srv, w.cap)), iters)
    grown = int((ctx_srv - w.ctx_lens).max().item())
    # bulk prefill encode: n_pre tokens of every sequence in one call (their own states, so
    # the cache is rewritten with the same bytes)
    n_pre = min(2048, ctx)
    pre = torch.empty(B, n_pre, 2, L, w.H, w.d, dtype=torch.bfloat16, device="cuda")
    rqm.synth_states(w.params, pre, pre.stride()[:5], 0, B, 0, n_pre, 0, L)
    t_pre = timeit(graph_of(lambda: rqm.encode_append(w.shape, w.cache, pre, pos_begin=0)), iters)
    pre_bytes = pre.numel() * 2
    del pre
    torch.cuda.empty_cache()
    clk = clocks.stop()

    # ---- end to end through the public API with host buffers ----
    # every step: the layers' queries and current-token states from pinned host memory,
    # and the layers' outputs back
    q_h = [lw.q.cpu().pin_memory() for lw in layers]
    p_h = [lw.pending.cpu().pin_memory() for lw in layers]
    o_h = [torch.empty(o.shape, dtype=o.dtype).pin_memory() for o in outs]

    def e2e_step():
        for lw, qh, ph in zip(layers, q_h, p_h):
            lw.q.copy_(qh, non_blocking=True)
            lw.pending.copy_(ph, non_blocking=True)
        step()
        for oh, o in zip(o_h, outs):
            oh.copy_(o, non_blocking=True)

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(args.steps):
        e2e_step()
    ev1.record(stream)
    torch.cuda.synchronize()
    t_e2e = ev0.elapsed_time(ev1) / args.steps
    h2d = sum(x.numel() * 2 for x in q_h + p_h)
    d2h = sum(x.numel() * 2 for x in o_h)

    # ---- bytes ----
    d, ng = cfg.head_dim, cfg.head_dim // 32
    ref_b = 2 * (d // 2 + 4 * ng)
    res_b = [2 * (d * b // 8 + 4 * ng + 2) for b in cfg.res_bits[: L - 1]]
    th = B * w.H * ctx                                   # token-heads of one layer
    io_b = w.q.numel() * 2 + w.pending.numel() * 2 + out.numel() * 2
    bytes_multi = th * (ref_b + sum(res_b)) + io_b
    bytes_per = th * (L * ref_b + sum(res_b)) + io_b
    bytes_bf16 = th * L * 2 * d * 2 + io_b
    kvtok = B * ctx * L                                  # per layer
    hbm, peak_kind = _peaks()

    def med(x):
        return statistics.median(x)

    dec_ms = med(t_dec)
    gbs = bytes_multi / (dec_ms * 1e-3) / 1e9
    breakdown = {
        "rq_decode_multiloop": {"ms": dec_ms, "kv_tokens_s": kvtok / (dec_ms * 1e-3),
                                "gbs": gbs, "frac_hbm_measured": gbs / hbm,
                                "frac_hbm_nominal_8tbs": gbs / 8000.0},
        "rq_decode_perloop": {"ms": med(t_per), "kv_tokens_s": kvtok / (med(t_per) * 1e-3),
                              "gbs": bytes_per / (med(t_per) * 1e-3) / 1e9,
                              "frac_hbm_measured": bytes_per / (med(t_per) * 1e-3) / 1e9 / hbm},
        "encode_append_us": 1e3 * med(t_enc),
    }
    if t_bf_multi:
        for name, tt in (("bf16_decode_multiloop", t_bf_multi), ("bf16_decode_perloop", t_bf_per)):
            m = med(tt)
            breakdown[name] = {"ms": m, "kv_tokens_s": kvtok / (m * 1e-3),
                               "gbs": bytes_bf16 / (m * 1e-3) / 1e9,
                               "frac_hbm_measured": bytes_bf16 / (m * 1e-3) / 1e9 / hbm}
        breakdown["speedup_vs_bf16"] = {"multiloop": med(t_bf_multi) / dec_ms,
                                        "perloop": med(t_bf_per) / med(t_per)}
    breakdown["storage_reduction_vs_bf16"] = 1 - (ref_b + sum(res_b)) / (L * 2 * d * 2)
    m = med(t_srv)
    breakdown["serving_step"] = {
        "what": "per-loop decode of all %d loops + encode of the token + ctx advance, one CUDA "
                "graph replayed %d times (ctx %d..%d)" % (L, len(t_srv), ctx, ctx + grown),
        "ms": m, "tokens_s": B / (m * 1e-3), "kv_tokens_s": kvtok / (m * 1e-3)}
    m = med(t_pre)
    breakdown["prefill_encode"] = {
        "what": "rq_encode_append of %d tokens x %d sequences in one call" % (n_pre, B),
        "ms": m, "tokens_s": B * n_pre / (m * 1e-3),
        "gbs": (pre_bytes + B * n_pre * w.H * (ref_b + sum(res_b))) / (m * 1e-3) / 1e9}
    if t_pg_multi:
        for name, tt, nb, base in (("rq_paged_decode_multiloop", t_pg_multi, bytes_multi, dec_ms),
                                   ("rq_paged_decode_perloop", t_pg_per, bytes_per, med(t_per))):
            m = med(tt)
            breakdown[name] = {"ms": m, "kv_tokens_s": kvtok / (m * 1e-3),
                               "gbs": nb / (m * 1e-3) / 1e9,
                               "frac_hbm_measured": nb / (m * 1e-3) / 1e9 / hbm,
                               "time_vs_contiguous": m / base}

    value = kvtok * NL * world / (ms * 1e-3)
    line = {
        "metric": METRIC, "value": value, "unit": "KV tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded Philox generator; no dataset)",
        "config": {"workload": _workload_desc(cfg), "step": "multi-loop decode attention + "
                   "deferred-write encode/append of the current token (CUDA graph replay)",
                   "layers_timed": NL,
                   "l2": "inputs larger than L2 (%.0f MB packed cache read per step)" %
                   (bytes_multi / 1e6), "parallelism": "replicas (weak, per-GPU batch %d)" % B},
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s",
                     "frac": gbs / hbm, "traffic": _traffic(cfg.name), "peak_kind": peak_kind,
                     "kernel": "rq_decode_attention (split kernel + combine, timed per call)",
                     "algorithmic_bytes_per_launch": bytes_multi},
        "cpu_baseline": cpu,
        "e2e": {"value": kvtok * NL * world / (t_e2e * 1e-3), "unit": "KV tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk,
        "breakdown": breakdown,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def budget_arm(args, cfg):
    """Fixed KV-memory budget per layer: the largest batch whose cache fits, for the packed
    cache and for the BF16 cache, and decode KV tokens/s of each at its own batch (one JSON
    line)."""
    import torch

    import looped_transformer_kv_gb300 as rqm
    from looped_transformer_kv_gb300.workload import Workload

    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
    budget = int(args.budget_gb * (1 << 30))
    cap = max(64, -(-(cfg.ctx + 2) // 64) * 64)
    L, H, d = cfg.n_loops, cfg.n_kv_heads, cfg.head_dim
    rq_seq = rqm.rq.cache_bytes(rqm.make_shape(1, cfg.n_q_heads, H, d, L, cap,
                                               cfg.res_bits[: L - 1]))
    bf_seq = 2 * H * L * cap * d * 2
    res = {"experiment": "fixed KV-memory budget per layer", "workload": _workload_desc(cfg),
           "budget_gib": args.budget_gb, "bytes_per_sequence": {"rq": rq_seq, "bf16": bf_seq}}
    iters = max(args.steps, 10)

    def timed(fn):
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            fn()
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr):
            fn()
        for _ in range(max(3, args.warmup)):
            gr.replay()
        torch.cuda.synchronize()
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        ev[0].record()
        for _ in range(iters):
            gr.replay()
        ev[1].record()
        torch.cuda.synchronize()
        return ev[0].elapsed_time(ev[1]) / iters

    for kind in ("rq", "bf16"):
        B = budget // (rq_seq if kind == "rq" else bf_seq)
        w = Workload(cfg, capacity=cap, batch=int(B), build_rq=kind == "rq",
                     build_bf16=kind == "bf16")
        out, ws = w.out_buffer(L), w.workspace(L)
        out1, ws1 = [w.out_buffer(1) for _ in range(L)], w.workspace(1)
        dec = w.decode if kind == "rq" else w.decode_bf16
        t_multi = timed(lambda: dec(0, L, out, ws))

        def per():
            for l in range(L):
                dec(l, 1, out1[l], ws1)

        t_per = timed(per)
        kvtok = B * cfg.ctx * L
        res[kind] = {"batch": int(B), "cache_gib": B * (rq_seq if kind == "rq" else bf_seq) / 2**30,
                     "multiloop_ms": t_multi, "multiloop_kv_tokens_s": kvtok / (t_multi * 1e-3),
                     "perloop_ms": t_per, "perloop_kv_tokens_s": kvtok / (t_per * 1e-3)}
        del w, out, ws, out1, ws1
        torch.cuda.empty_cache()
    res["batch_ratio"] = res["rq"]["batch"] / res["bf16"]["batch"]
    res["throughput_ratio_multiloop"] = (res["rq"]["multiloop_kv_tokens_s"] /
                                         res["bf16"]["multiloop_kv_tokens_s"])
    res["throughput_ratio_perloop"] = (res["rq"]["perloop_kv_tokens_s"] /
                                       res["bf16"]["perloop_kv_tokens_s"])
    print(json.dumps(res), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default="layer_1p4b")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-bf16", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-paged", action="store_true")
    ap.add_argument("--budget-gb", type=float, default=0.0,
                    help="run the fixed KV-memory budget experiment (GiB per layer) instead")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    import synth
    cfg = synth.config_by_name(args.workload)
    if args.impl == "reference":
        reference_arm(args, cfg)
    else:
        from __graft_entry__ import build
        build()
        if args.budget_gb > 0:
            budget_arm(args, cfg)
        else:
            gpu_arm(args, cfg)


if __name__ == "__main__":
    main()
