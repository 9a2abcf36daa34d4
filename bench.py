#!/usr/bin/env python
"""Decode-attention benchmark of librq on one GB300 (one JSON line on stdout).

A step is one decode step of one layer of a looped model on the workload's batch: fused
decode attention of every loop over the packed cache (all loops' queries in one call, the
reference tile read once) plus the deferred write of the current token (encode + append of
its L loop states).  Metric: KV tokens/s = batch * ctx * loops * layers / step time.

The headline workload is the serving-scale one (B 128, ctx 32768, 16 heads, d 128, 4 loops,
decode and deferred-write encode interleaved in a step).  The line's `breakdown` also carries,
measured in the same run, every other workload (per-layer times, all 24 layers for mixed_24l),
the BF16 comparison kernel on the same shapes, the paged cache, the serving step under a CUDA
graph, the bulk prefill encode, the fixed KV-memory budget experiment and the ablation rows
(per-loop throughput of the method with a fixed at 1 and of direct quantisation).

python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]
                [--no-sweep] [--no-bf16] [--no-paged] [--no-cpu-baseline] [--budget-gb G]

With --gpus N > 1 (launched by torch.distributed.run) every rank runs the whole workload on
its own GPU (independent sequences: weak scaling, no collective on the data path); times
are max-reduced over ranks.  --impl reference times the fp64 CPU oracle on the host cores.
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
# of the split kernel, from one ncu capture, keyed by the kernel sources they were taken on;
# any change to those sources makes the figure stale (reported as null).
KERNEL_SOURCES = ("looped_transformer_kv_gb300/csrc/rq_decode_mma.cu",
                  "looped_transformer_kv_gb300/csrc/rq_decode_mma.cuh",
                  "looped_transformer_kv_gb300/csrc/rq_ptx.cuh",
                  "looped_transformer_kv_gb300/csrc/rq_common.cuh",
                  "looped_transformer_kv_gb300/csrc/rq_kernels.h")
TRAFFIC = {
    # serving all-loops split kernel, one launch: 30.87 GB read + 19.68 MB written (ncu, 1 pass)
    ("3a7e1d92a5201883", "serving"): 30870000000 + 19680000,
}


def _kernel_hash():
    import hashlib
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def _traffic(workload):
    return TRAFFIC.get((_kernel_hash(), workload))


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
#
# The fp64 oracle's decode (rotated form) of all loops, timed on its own: slices of the
# workload (one sequence and kv-head each) are generated and encoded first (untimed), then
# every worker process -- one per host core, one BLAS thread each -- decodes its slices in
# rounds that start together; a round's wall clock is taken between two barriers.

_BLAS_ENV = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")


def _oracle_worker(name, slices, rounds, barrier, results):
    import numpy as np

    import oracle as O
    import synth
    cfg = synth.config_by_name(name)
    rb = cfg.res_bits[: cfg.n_loops - 1]
    g = cfg.n_q_heads // cfg.n_kv_heads
    signs = synth.rotation_signs(cfg, 0)
    prepared = []
    for b, h in slices:
        x = synth.gen_states(cfg, 0, [b], np.arange(cfg.ctx + 1), heads=[h])[0, :, :, :, 0, :]
        x = x.astype(np.float64)
        s = signs[h].astype(np.float64)
        ek = O.encode(x[:cfg.ctx, 0], s[0], rb)
        ev = O.encode(x[:cfg.ctx, 1], s[1], rb)
        q = synth.gen_queries(cfg, 0, [b])[0, h * g:(h + 1) * g].astype(np.float64)
        prepared.append((ek, ev, s, q, x[cfg.ctx]))
    barrier.wait()                                  # every worker's slices are ready
    for _ in range(rounds):
        barrier.wait()                              # round start
        for ek, ev, s, q, pend in prepared:
            for l in range(cfg.n_loops):
                O.decode_rotated(q[:, l], ek, ev, s[0], s[1], l, pend[0, l], pend[1, l])
        barrier.wait()                              # round end
    results.put(len(prepared))


def run_oracle(name, n_workers, per_worker, rounds):
    """Round wall-clock times (s) of the oracle decode on n_workers processes, each with
    per_worker slices spread over the batch and heads; returns (times, kv_tokens_per_round,
    description of the sample)."""
    import multiprocessing as mp

    import synth
    cfg = synth.config_by_name(name)
    units = [(b, h) for b in range(cfg.batch) for h in range(cfg.n_kv_heads)]
    n = min(len(units), n_workers * per_worker)
    stride = len(units) / n
    chosen = [units[int(i * stride)] for i in range(n)]
    work = [chosen[i::n_workers] for i in range(n_workers)]
    work = [w for w in work if w]
    saved = {k: os.environ.get(k) for k in _BLAS_ENV}
    for k in _BLAS_ENV:
        os.environ[k] = "1"
    ctx = mp.get_context("spawn")
    barrier = ctx.Barrier(len(work) + 1)
    results = ctx.Queue()
    procs = [ctx.Process(target=_oracle_worker, args=(name, w, rounds, barrier, results))
             for w in work]
    try:
        for p in procs:
            p.start()
        barrier.wait(timeout=1800)                  # slices generated and encoded
        times = []
        for _ in range(rounds):
            barrier.wait(timeout=1800)
            t0 = time.perf_counter()
            barrier.wait(timeout=1800)
            times.append(time.perf_counter() - t0)
        done = sum(results.get(timeout=600) for _ in procs)
        for p in procs:
            p.join(timeout=600)
    finally:
        for p in procs:
            if p.is_alive():
                p.terminate()
        for k, v in saved.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
    assert done == n
    tokens = n * cfg.ctx * cfg.n_loops
    desc = ("%d of the %d (sequence, kv-head) slices, spread over the batch, each: fp64 oracle "
            "decode (rotated form) of all %d loops over ctx %d; %d worker process(es), one "
            "BLAS thread each" % (n, len(units), cfg.n_loops, cfg.ctx, len(work)))
    return times, tokens, desc


def cpu_baseline(name, rounds=3):
    """All host cores over a fraction of the slices, and one core on one slice."""
    cores = os.cpu_count() or 1
    t1, tok1, _ = run_oracle(name, 1, 1, rounds)
    single = tok1 / statistics.median(t1)
    tn, tokn, desc = run_oracle(name, cores, 1, rounds)
    value = tokn / statistics.median(tn)
    return {"value": value, "unit": "KV tokens/s", "cores": cores, "kind": "oracle",
            "sample": desc + "; median of %d rounds" % rounds,
            "single_thread": {"value": single, "unit": "KV tokens/s",
                              "sample": "one slice, one process, one BLAS thread"}}


def reference_arm(args, cfg):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    cores = os.cpu_count() or 1
    times, tok, desc = run_oracle(cfg.name, cores, 1, args.warmup + args.steps)
    times = times[args.warmup:]
    t = sum(times)
    value = tok * len(times) / t
    sample = desc + "; a step is one round over the sampled slices"
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


def graph_of(fn):
    """Capture fn (a sequence of library calls on the current stream) in a CUDA graph."""
    import torch
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


def timeit(gr, iters, warmup=3):
    """Per-replay device times (ms) of a captured graph, CUDA events on the current stream."""
    import torch
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        gr.replay()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(iters + 1)]
    torch.cuda.synchronize()
    ev[0].record(stream)
    for i in range(iters):
        gr.replay()
        ev[i + 1].record(stream)
    torch.cuda.synchronize()
    return [ev[i].elapsed_time(ev[i + 1]) for i in range(iters)]


def byte_counts(cfg, w, out):
    """Algorithmic bytes of one layer's decode call: all-loops, per-loop (sum of the L calls)
    and the BF16 kernel, each with the queries, current token and outputs."""
    L, d = cfg.n_loops, cfg.head_dim
    ng = d // 32
    ref_b = 2 * (d // 2 + 4 * ng)
    res_b = [2 * (d * b // 8 + 4 * ng + 2) for b in cfg.res_bits[: L - 1]]
    th = w.B * w.H * cfg.ctx
    io_b = w.q.numel() * 2 + w.pending.numel() * 2 + out.numel() * 2
    return {"multi": th * (ref_b + sum(res_b)) + io_b,
            "per": th * (L * ref_b + sum(res_b)) + io_b,
            "bf16": th * L * 2 * d * 2 + io_b,
            "per_token_head_multi": ref_b + sum(res_b), "ref_b": ref_b, "res_b": res_b}


def _row(ms, kvtok, nbytes, hbm):
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {"ms": ms, "kv_tokens_s": kvtok / (ms * 1e-3), "gbs": gbs, "frac_hbm_measured": gbs / hbm,
            "frac_hbm_nominal_8tbs": gbs / 8000.0}


def decode_timings(w, iters, bf16, L):
    """Graph-replayed per-call times (ms, medians) of workload w's all-loops and per-loop
    decode calls, and of the BF16 kernel's on the same shapes if built."""
    med = statistics.median
    out, ws, ws1 = w.out_buffer(L), w.workspace(L), w.workspace(1)
    out1 = [w.out_buffer(1) for _ in range(L)]
    t = {"multi": med(timeit(graph_of(lambda: w.decode(0, L, out, ws)), iters))}

    def per():
        for l in range(L):
            w.decode(l, 1, out1[l], ws1)

    t["per"] = med(timeit(graph_of(per), iters))
    if bf16:
        t["bf16_multi"] = med(timeit(graph_of(lambda: w.decode_bf16(0, L, out, ws)), iters))

        def bf_per():
            for l in range(L):
                w.decode_bf16(l, 1, out1[l], ws1)

        t["bf16_per"] = med(timeit(graph_of(bf_per), iters))
    return t, out


def workload_rows(cfg, nb, t, hbm, layers=1):
    """Breakdown rows of one workload from its per-layer times (t: decode_timings) and byte
    counts (nb: byte_counts)."""
    L = cfg.n_loops
    kvtok = cfg.batch * cfg.ctx * L
    rows = {"rq_decode_multiloop": _row(t["multi"], kvtok, nb["multi"], hbm),
            "rq_decode_perloop": _row(t["per"], kvtok, nb["per"], hbm)}
    if "bf16_multi" in t:
        rows["bf16_decode_multiloop"] = _row(t["bf16_multi"], kvtok, nb["bf16"], hbm)
        rows["bf16_decode_perloop"] = _row(t["bf16_per"], kvtok, nb["bf16"], hbm)
        rows["speedup_vs_bf16"] = {"multiloop": t["bf16_multi"] / t["multi"],
                                   "perloop": t["bf16_per"] / t["per"]}
    if layers > 1:
        rows["layers"] = layers
        rows["note"] = ("times are per layer (mean over all %d layers, each timed on its own "
                        "cache); BF16 timed on layer 0" % layers)
    return rows


def sweep_workload(name, iters, hbm):
    """Another workload at full size: all-loops and per-loop decode per layer, the BF16
    kernel on the same shapes; multi-layer workloads time every layer in turn (each layer's
    cache built, timed and freed)."""
    import torch

    import synth
    from looped_transformer_kv_gb300.workload import Workload
    cfg = synth.config_by_name(name)
    L = cfg.n_loops
    tm, tp = [], []
    t0 = nb = None
    for layer in range(cfg.layers):
        w = Workload(cfg, layer=layer, capacity=cfg.ctx + 2, build_bf16=(layer == 0))
        t, out = decode_timings(w, iters, layer == 0, L)
        tm.append(t["multi"])
        tp.append(t["per"])
        if layer == 0:
            t0, nb = t, byte_counts(cfg, w, out)
        del w, out
        torch.cuda.empty_cache()
    t = dict(t0)
    t["multi"] = statistics.mean(tm)
    t["per"] = statistics.mean(tp)
    rows = workload_rows(cfg, nb, t, hbm, cfg.layers)
    rows["workload"] = _workload_desc(cfg)
    if cfg.layers > 1:
        rows["model_step_ms"] = {"multiloop": sum(tm), "perloop": sum(tp)}
        rows["layer_ms_range"] = {"multiloop": [min(tm), max(tm)], "perloop": [min(tp), max(tp)]}
    return rows


def budget_experiment(name, budget_gib, iters):
    """Fixed KV-memory budget per layer: the largest batch whose cache fits, for the packed and
    for the BF16 cache, and decode KV tokens/s of each at its own batch."""
    import torch

    import synth
    from looped_transformer_kv_gb300.workload import Workload, budget_batches
    cfg = synth.config_by_name(name)
    budget = int(budget_gib * (1 << 30))
    cap = max(64, -(-(cfg.ctx + 2) // 64) * 64)
    L = cfg.n_loops
    b_rq, b_bf, rq_seq, bf_seq = budget_batches(cfg, budget, cap)
    res = {"experiment": "fixed KV-memory budget per layer", "workload": _workload_desc(cfg),
           "budget_gib": budget_gib, "bytes_per_sequence": {"rq": rq_seq, "bf16": bf_seq}}
    med = statistics.median
    for kind, B in (("rq", b_rq), ("bf16", b_bf)):
        w = Workload(cfg, capacity=cap, batch=int(B), build_rq=kind == "rq",
                     build_bf16=kind == "bf16")
        out, ws = w.out_buffer(L), w.workspace(L)
        out1, ws1 = [w.out_buffer(1) for _ in range(L)], w.workspace(1)
        dec = w.decode if kind == "rq" else w.decode_bf16
        t_multi = med(timeit(graph_of(lambda: dec(0, L, out, ws)), iters))

        def per():
            for l in range(L):
                dec(l, 1, out1[l], ws1)

        t_per = med(timeit(graph_of(per), iters))
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
    return res


def ablation_rows(name, iters, hbm):
    """Ablation rows of the method's steps (include/rq_ablation.h), on one workload: each
    variant's cache is encoded with its own a (least squares / 1 / 0) and decoded by causal
    per-loop calls (loop l < L-1 by the variant's kernel, the final loop, the INT4 reference,
    by the method's kernel); bytes are what each variant's decode reads."""
    import torch

    import synth
    from looped_transformer_kv_gb300.workload import Workload
    cfg = synth.config_by_name(name)
    L, d = cfg.n_loops, cfg.head_dim
    ng = d // 32
    ref_b = 2 * (d // 2 + 4 * ng)
    res_b = [2 * (d * b // 8 + 4 * ng) for b in cfg.res_bits[: L - 1]]   # codes + step/offset
    rows = {"workload": _workload_desc(cfg),
            "what": "all L loops as causal per-loop calls; bytes = what each decode reads"}
    med = statistics.median
    for variant, mode in (("rq", 0), ("a_one", 1), ("direct_rotated", 2)):
        w = Workload(cfg, capacity=cfg.ctx + 2, alpha_mode=mode)
        outs = [w.out_buffer(1) for _ in range(L)]
        ws1 = w.workspace(1)

        def per():
            for l in range(L):
                if mode == 0 or l == L - 1:
                    w.decode(l, 1, outs[l], ws1)
                else:
                    w.decode_ablation(l, outs[l], ws1)

        t = med(timeit(graph_of(per), iters))
        a_b = 0 if mode else 4                               # the a stream (K and V)
        per_th = sum((ref_b if mode != 2 else 0) + rb + a_b for rb in res_b) + ref_b
        th = w.B * w.H * cfg.ctx
        nbytes = th * per_th + w.q.numel() * 2 + w.pending.numel() * 2 + outs[0].numel() * 2 * L
        rows[variant] = dict(_row(t, w.B * cfg.ctx * L, nbytes, hbm), bytes_per_token_head=per_th)
        del w, outs, ws1
        torch.cuda.empty_cache()
    return rows


def gpu_arm(args, cfg):
    import torch
    import torch.distributed as dist

    import looped_transformer_kv_gb300 as rqm
    from looped_transformer_kv_gb300.workload import Workload

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        # the oracle runs in spawned processes before this one touches the GPU
        cpu = cpu_baseline(cfg.name)

    if world > 1:
        dist.init_process_group("gloo")
    torch.cuda.set_device(local)

    # spare slots past ctx: the deferred write of the current token lands in slot ctx,
    # which the step's attention (ctx_lens = ctx) does not read, so every step is the same.
    # Every layer of the model gets its own packed cache (the BF16 cache of one layer is
    # built for the comparison kernel: the same shapes for every layer).
    layers = [Workload(cfg, layer=l, capacity=cfg.ctx + 2, build_bf16=(l == 0 and not args.no_bf16))
              for l in range(cfg.layers)]
    w = layers[0]
    NL = len(layers)
    L, B, ctx = cfg.n_loops, w.B, cfg.ctx
    ws = w.workspace(L)
    outs = [lw.out_buffer(L) for lw in layers]
    # deferred write of the current token: its L states, appended at slot ctx
    pos_new = torch.full((B, 1), ctx, dtype=torch.int32, device="cuda")

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

    g_step = graph_of(step)
    # ---- warm-up, then the timed steps (barrier + synchronize on both sides) ----
    for _ in range(args.warmup):
        g_step.replay()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clocks = Clocks(local)
    time.sleep(0.3)
    stream = torch.cuda.current_stream()
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

    # ---- per-call timings of the headline workload (graph replays, CUDA events) ----
    iters = max(args.steps, 20)
    med = statistics.median
    hbm, peak_kind = _peaks()
    t, out = decode_timings(w, iters, not args.no_bf16, L)
    new_kv = w.pending.reshape(B, 1, 2, L, w.H, w.d)
    t_enc = timeit(graph_of(lambda: rqm.encode_append(w.shape, w.cache, new_kv, positions=pos_new)),
                   iters)
    nb = byte_counts(cfg, w, out)
    breakdown = workload_rows(cfg, nb, t, hbm)
    breakdown["encode_append_us"] = 1e3 * med(t_enc)
    breakdown["interleaved_step_ms"] = ms / NL
    breakdown["storage_reduction_vs_bf16"] = 1 - nb["per_token_head_multi"] / (L * 2 * cfg.head_dim * 2)
    out1 = [w.out_buffer(1) for _ in range(L)]
    ws1 = w.workspace(1)
    # the same tokens in a paged cache (64-token pages scattered over a pool with spare pages)
    if not args.no_paged:
        pc, paging, bt = w.paged_twin(spare_pages=64, seed=1)
        t_pg_multi = med(timeit(graph_of(lambda: w.decode_paged(pc, paging, 0, L, out, ws)), iters))

        def pg_per():
            for l in range(L):
                w.decode_paged(pc, paging, l, 1, out1[l], ws1)

        t_pg_per = med(timeit(graph_of(pg_per), iters))
        kvtok = B * ctx * L
        for name, tt, nbytes, base in (("rq_paged_decode_multiloop", t_pg_multi, nb["multi"], t["multi"]),
                                       ("rq_paged_decode_perloop", t_pg_per, nb["per"], t["per"])):
            breakdown[name] = _row(tt, kvtok, nbytes, hbm)
            breakdown[name]["time_vs_contiguous"] = tt / base
        del pc, paging, bt
        torch.cuda.empty_cache()
    # serving step: the L per-loop decode calls, the deferred write of the token into slot
    # ctx_len and the advance of ctx_len, captured once and replayed token after token (the
    # spare capacity past ctx takes the appended tokens)
    ctx_srv = w.ctx_lens.clone()
    ws_srv = w.workspace_for(1, w.cap)
    t_srv = timeit(graph_of(lambda: w.serving_step(ctx_srv, out1, ws_srv, w.cap)), iters, warmup=0)
    grown = int((ctx_srv - w.ctx_lens).max().item())
    m = med(t_srv)
    breakdown["serving_step"] = {
        "what": "per-loop decode of all %d loops + encode of the token + ctx advance, one CUDA "
                "graph replayed %d times (ctx %d..%d)" % (L, len(t_srv), ctx, ctx + grown),
        "ms": m, "tokens_s": B / (m * 1e-3), "kv_tokens_s": B * ctx * L / (m * 1e-3)}
    # bulk prefill encode: n_pre tokens of every sequence in one call (their own states, so
    # the cache is rewritten with the same bytes)
    n_pre = min(2048, ctx)
    bpre = min(B, 16)
    pre = torch.empty(bpre, n_pre, 2, L, w.H, w.d, dtype=torch.bfloat16, device="cuda")
    rqm.synth_states(w.params, pre, pre.stride()[:5], 0, bpre, 0, n_pre, 0, L)
    sub = w._sub_cache(0, bpre)
    sub_shape = rqm.make_shape(bpre, w.Hq, w.H, w.d, L, w.cap, cfg.res_bits[: L - 1])
    t_pre = timeit(graph_of(lambda: rqm.encode_append(sub_shape, sub, pre, pos_begin=0)), iters)
    m = med(t_pre)
    breakdown["prefill_encode"] = {
        "what": "rq_encode_append of %d tokens x %d sequences in one call" % (n_pre, bpre),
        "ms": m, "tokens_s": bpre * n_pre / (m * 1e-3),
        "gbs": (pre.numel() * 2 + bpre * n_pre * w.H * nb["per_token_head_multi"]) / (m * 1e-3) / 1e9}
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

    kvtok = B * ctx * L                                  # per layer
    dec = breakdown["rq_decode_multiloop"]
    value = kvtok * NL * world / (ms * 1e-3)
    del layers, outs, out, out1, w, g_step, ws, ws1, ws_srv
    torch.cuda.empty_cache()

    # ---- every other workload and the fixed-budget experiment, measured in this run ----
    if world == 1 and not args.no_sweep:
        import synth
        per = {}
        for other in synth.CONFIGS:
            if other.name != cfg.name:
                per[other.name] = sweep_workload(other.name, iters, hbm)
        breakdown["per_workload"] = per
    if world == 1 and not args.no_sweep:
        breakdown["ablation"] = ablation_rows("layer_1p4b", iters, hbm)
    if world == 1 and args.budget_gb > 0:
        breakdown["budget"] = budget_experiment(args.budget_workload, args.budget_gb,
                                                max(10, args.steps))

    line = {
        "metric": METRIC, "value": value, "unit": "KV tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded Philox generator; no dataset)",
        "config": {"workload": _workload_desc(cfg), "step": "multi-loop decode attention + "
                   "deferred-write encode/append of the current token (CUDA graph replay)",
                   "layers_timed": NL,
                   "l2": "inputs larger than L2 (%.0f MB packed cache read per step)" %
                   (nb["multi"] / 1e6), "parallelism": "replicas (weak, per-GPU batch %d)" % B},
        "roofline": {"bound": "hbm", "achieved": dec["gbs"], "peak": hbm, "unit": "GB/s",
                     "frac": dec["gbs"] / hbm, "traffic": _traffic(cfg.name),
                     "peak_kind": peak_kind,
                     "kernel": "rq_decode_attention all-loops call (split kernel + combine, "
                               "timed per call)",
                     "algorithmic_bytes_per_launch": nb["multi"]},
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


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default="serving")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-bf16", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-paged", action="store_true")
    ap.add_argument("--no-sweep", action="store_true",
                    help="skip the other workloads and the budget experiment")
    ap.add_argument("--budget-gb", type=float, default=8.0,
                    help="fixed KV-memory budget per layer (GiB) of the budget experiment; 0: skip")
    ap.add_argument("--budget-workload", default="layer_1p4b")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    if args.no_sweep:
        args.budget_gb = 0.0
    import synth
    cfg = synth.config_by_name(args.workload)
    if args.impl == "reference":
        reference_arm(args, cfg)
    else:
        from __graft_entry__ import build
        build()
        gpu_arm(args, cfg)


if __name__ == "__main__":
    main()
