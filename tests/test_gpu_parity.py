"""GPU parity: librq (through its C ABI) against the fp64 oracle on seeded inputs."""

import dataclasses

import numpy as np
import pytest

import oracle as O
import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import looped_transformer_kv_gb300 as rqm
    from looped_transformer_kv_gb300.workload import Workload, slice_from_records

from rq_parity import check_slice, Follow, gpu_slice_to_oracle_names, packed_bytes_equal  # noqa: E402


def _cfg(name, **kw):
    return dataclasses.replace(synth.config_by_name(name), **kw)


# ------------------------------------------------------------------ generator twins

@pytest.mark.parametrize("name", ["pr1_small", "gqa_deep", "mixed_24l"])
def test_gpu_generator_matches_host_generator(name):
    cfg = synth.config_by_name(name)
    w = Workload(cfg, capacity=64, ctx_lens=[40] * 2, batch=2, build_rq=False)
    buf = torch.empty(2, 64, 2, cfg.n_loops, cfg.n_kv_heads, cfg.head_dim,
                      dtype=torch.bfloat16, device="cuda")
    rqm.synth_states(w.params, buf, buf.stride()[:5], 0, 2, 0, 64, 0, cfg.n_loops)
    host = synth.gen_states(cfg, 0, [0, 1], np.arange(64))          # [b][t][kv][l][h][d]
    gpu = buf.float().cpu().numpy()
    assert np.array_equal(gpu, host)
    qh = synth.gen_queries(cfg, 0, [0, 1])
    assert np.array_equal(w.q.float().cpu().numpy(), qh)


# ------------------------------------------------------------------ small shapes

SMALL = [
    # name, overrides, ctx_lens
    ("pr1_small", {}, [256]),
    ("layer_1p4b", dict(batch=3, n_q_heads=2, n_kv_heads=2), [257, 33, 1]),
    ("mixed_24l", dict(batch=2, n_q_heads=2, n_kv_heads=2), [100, 0]),
    ("gqa_deep", dict(batch=3, n_q_heads=8, n_kv_heads=2), [31, 32, 2]),
    ("layer_1p4b", dict(batch=1, n_q_heads=4, n_kv_heads=4, n_loops=1, res_bits=()), [70]),
    ("pr1_small", dict(n_loops=2, res_bits=(4,), sigma=(0.3, 0.1)), [300]),
    ("pr1_small", dict(n_q_heads=8, n_kv_heads=2, n_loops=8, res_bits=(2, 4) * 3 + (2,),
                       sigma=(0.1,) * 8), [129]),
]


@pytest.mark.parametrize("case", range(len(SMALL)))
@pytest.mark.parametrize("pending", [True, False])
def test_small_parity(case, pending):
    name, over, ctx = SMALL[case]
    cfg = _cfg(name, **over)
    cap = max(ctx) + 2
    w = Workload(cfg, capacity=cap, ctx_lens=ctx, batch=len(ctx))
    calls, outs, wss = [], [], []

    def call(l0, lc):
        o, ws = w.out_buffer(lc), w.workspace(lc)
        w.decode(l0, lc, o, ws, pending=pending)
        calls.append((l0, lc))
        outs.append(o)
        wss.append(ws)

    for l in range(cfg.n_loops):                       # causal per-loop calls
        call(l, 1)
    call(0, cfg.n_loops)                               # all loops in one call
    if cfg.n_loops > 2:                                # a middle range
        call(1, 2)
    torch.cuda.synchronize()
    for ws in wss:                                     # no pipeline wait gave up
        assert ws[:1].view(torch.int32).item() == 0
    for b in range(len(ctx)):
        for h in range(cfg.n_kv_heads):
            check_slice(w, b, h, calls, outs, pending=pending)
    # the multi-loop call and the per-loop calls compute the same attention
    per = torch.cat(outs[: cfg.n_loops], dim=2).float()
    assert torch.allclose(per, outs[cfg.n_loops].float(), atol=2e-3, rtol=1e-2)


# ------------------------------------------------------------------ seeded random shapes

def _random_case(seed):
    """A small shape drawn from the ranges the library supports (head dim 64/128, 1-8 query
    heads per kv-head, 1-8 loops with 2- and 4-bit residual loops, ragged contexts), the
    generator's parameters drawn as well; calls: every loop alone, all loops, a random range."""
    rng = np.random.default_rng(1000 + seed)
    d = int(rng.choice([64, 128]))
    g = int(rng.choice([1, 2, 4, 8]))
    H = int(rng.integers(1, 4))
    L = int(rng.integers(1, 9))
    B = int(rng.integers(1, 4))
    res_bits = tuple(int(rng.choice([2, 4])) for _ in range(L - 1))
    sigma = tuple(float(np.float32(rng.uniform(0.03, 0.3))) for _ in range(L))
    cfg = synth.Config(f"random{seed}", 1, B, g * H, H, d, L, 512, res_bits,
                       int(rng.integers(0, 4)), float(rng.choice([4.0, 8.0, 16.0])), sigma,
                       int(rng.integers(0, 2)), int(rng.integers(0, 1 << 20)))
    ctx = [int(rng.choice([0, 1, 63, 64, 65, 128, 191, 257, 300, 384, 447])) for _ in range(B)]
    lb = int(rng.integers(0, L))
    lc = int(rng.integers(1, L - lb + 1))
    return cfg, ctx, (lb, lc), bool(rng.integers(0, 2))


@pytest.mark.parametrize("seed", range(16))
def test_random_shapes_parity(seed):
    cfg, ctx, extra, pending = _random_case(seed)
    w = Workload(cfg, capacity=max(ctx) + 2, ctx_lens=ctx, batch=len(ctx))
    calls = [(l, 1) for l in range(cfg.n_loops)] + [(0, cfg.n_loops), extra]
    outs, wss = [], []
    for l0, lc in calls:
        o, ws = w.out_buffer(lc), w.workspace(lc)
        w.decode(l0, lc, o, ws, pending=pending)
        outs.append(o)
        wss.append(ws)
    torch.cuda.synchronize()
    for ws in wss:
        assert ws[:1].view(torch.int32).item() == 0
    for b in range(len(ctx)):
        for h in range(cfg.n_kv_heads):
            check_slice(w, b, h, calls, outs, pending=pending)


# ------------------------------------------------------------------ degenerate inputs

def _encode_custom(x, d, L, res_bits, signs):
    """Encode host states x [N][2][L][d] (bf16 values) through librq; returns the slice."""
    N = x.shape[0]
    cap = -(-N // 64) * 64
    shape = rqm.make_shape(1, 1, 1, d, L, cap, res_bits)
    cache = rqm.PackedCache(shape, torch.from_numpy(signs[:, None, :].copy()))
    kv = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).cuda()
    kv = kv.reshape(1, N, 2, L, 1, d)
    rqm.encode_append(shape, cache, kv, pos_begin=0)
    torch.cuda.synchronize()
    # the N encoded slots (N even: whole V token pairs)
    sl = slice_from_records(cache, cache.records()[0, 0, :cap // 64], N)
    return sl, cap


@pytest.mark.parametrize("d", [64, 128])
def test_degenerate_groups_encode(d):
    rng = np.random.default_rng(0)
    L, res_bits = 4, [2, 4, 2]
    N = 8
    x = O.bf16_round(rng.standard_normal((N, 2, L, d)))
    x[0] = 0.0                                           # all zero token
    x[1, :, :, :32] = 0.75                               # constant group in every loop
    x[2, :, :, :] = x[2, :, L - 1:L, :]                  # all loops equal the reference
    x[3, 1, :, 5] = 40.0                                 # outlier channel
    x[4, :, :L - 1] = 0.0                                # zero residual loops, nonzero ref
    x[5, :, L - 1] = 0.0                                 # zero reference: a = 0
    signs = np.where(rng.random((2, d)) < 0.5, -1, 1).astype(np.int8)
    sl, _ = _encode_custom(x, d, L, res_bits, signs)
    for kv in range(2):
        f = Follow(gpu_slice_to_oracle_names(sl, kv, d, L, res_bits))
        enc = O.encode(x[:, kv], signs[kv].astype(np.float64), res_bits, rnd=f)
        assert f.bad == 0, f.bad_names
        assert packed_bytes_equal(enc, sl, kv, res_bits)
    assert np.all(sl[("alpha", 0, 0)][5] == 0.0)


def test_on_grid_reference_gives_zero_residual_on_gpu():
    rng = np.random.default_rng(4)
    d, L, N = 128, 4, 6
    codes = rng.integers(0, 16, size=(N, d // 32, 32))
    codes[:, :, 0], codes[:, :, 1] = 0, 15
    s = 2.0 ** rng.integers(-5, 0, size=(N, d // 32, 1))
    ref = (codes * s + rng.integers(-8, 2, size=(N, d // 32, 1)) * s).reshape(N, d)
    x = np.repeat(np.repeat(ref[:, None, None, :], 2, axis=1), L, axis=2)
    signs = np.where(rng.random((2, d)) < 0.5, -1, 1).astype(np.int8)
    sl, _ = _encode_custom(x, d, L, [2, 2, 2], signs)
    for kv in range(2):
        for l in range(L - 1):
            assert np.all(sl[("alpha", kv, l)][:N] == 1.0)
            assert np.all(sl[("res_codes", kv, l)][:N] == 0)
            assert np.all(sl[("res_meta", kv, l)][:N] == 0.0)


# ------------------------------------------------------------------ BF16 comparison kernel

@pytest.mark.parametrize("name,over,ctx", [
    ("pr1_small", {}, [256]),
    ("gqa_deep", dict(batch=2, n_q_heads=8, n_kv_heads=2), [300, 5]),
])
def test_bf16_kernel_matches_textbook_attention(name, over, ctx):
    cfg = _cfg(name, **over)
    w = Workload(cfg, capacity=max(ctx) + 2, ctx_lens=ctx, batch=len(ctx), build_rq=False,
                 build_bf16=True)
    o = w.out_buffer(cfg.n_loops)
    w.decode_bf16(0, cfg.n_loops, o, w.workspace(cfg.n_loops))
    torch.cuda.synchronize()
    got = o.float().cpu().numpy()
    g = cfg.n_q_heads // cfg.n_kv_heads
    for b, c in enumerate(ctx):
        x = synth.gen_states(cfg, 0, [b], np.arange(c + 1))[0].astype(np.float64)  # [t][kv][l][h][d]
        q = synth.gen_queries(cfg, 0, [b])[0].astype(np.float64)
        for hq in range(cfg.n_q_heads):
            h = hq // g
            for l in range(cfg.n_loops):
                ref = O.softmax_attention(q[hq, l][None], x[:, 0, l, h], x[:, 1, l, h],
                                          1 / np.sqrt(cfg.head_dim))[0]
                e = np.abs(got[b, hq, l] - ref)
                from rq_parity import bf16_half_ulp
                assert np.max(e - bf16_half_ulp(ref)) <= 2e-3


# ------------------------------------------------------------------ status codes

def test_invalid_calls_return_status_and_enqueue_nothing():
    cfg = _cfg("pr1_small")
    w = Workload(cfg, capacity=64, ctx_lens=[10], batch=1)
    o = w.out_buffer(1)
    small = torch.empty(1, dtype=torch.float32, device="cuda")
    with pytest.raises(rqm.rq._lib.RqError) as e:
        w.decode(0, 1, o, small)
    assert e.value.status == 3
    with pytest.raises(rqm.rq._lib.RqError) as e:
        w.decode(3, 2, o, w.workspace(2))
    assert e.value.status == 1
