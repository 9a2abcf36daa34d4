"""Synthetic looped K/V states and queries for the five ResidualQuant workloads.

Workloads (all single-GPU, bf16 inputs, group 32, INT4 reference):
  pr1_small   1 layer,  B 1,   Hq=Hkv=2,   d 64,  4 loops, ctx 256,   residual bits 2,2,2
  layer_1p4b  1 layer,  B 16,  Hq=Hkv=16,  d 128, 4 loops, ctx 4096,  residual bits 2,2,2
  mixed_24l   24 layers, B 64, Hq=Hkv=16,  d 128, 4 loops, ctx 8192,  residual bits 4,2,2
  gqa_deep    1 layer,  B 32,  Hq 32/Hkv 8, d 128, 8 loops, ctx 16384, residual bits 2 x7
  serving     1 layer,  B 128, Hq=Hkv=16,  d 128, 4 loops, ctx 32768, residual bits 2,2,2

State model (looped Transformer: every loop of the shared block makes its own K/V, and
the loops' states are highly similar -- "ResidualQuant: KV Cache Quantization for Looped
Transformers with 2-Bit Residuals", abstract):
    x[b, t, kv, l, h, i] = bf16( u_l * base[b, t, kv, h, i] + sigma_l * n[b, t, kv, l, h, i] )
with base ~ N(0, 1) (Student-t with 3 degrees of freedom for gqa_deep), a fixed set of
outlier channels per (layer, kv-head, K/V) multiplied by a constant, u_l ~ U(0.8, 1.2) per
(token, head, loop, K/V), n ~ N(0, 1).  Queries are bf16 N(0, 1).

Normal draws are the Irwin-Hall sum of twelve 10-bit uniforms taken from one Philox block,
minus 6 (mean 0, variance 1 - 2^-20, support [-6, 6]); every operation after the integer
sum is an exactly specified IEEE fp32 operation, so the CUDA twin reproduces each value
bit for bit.

Philox counter layout (key = (seed & 0xffffffff, seed >> 32)):
    c0 = token position (or decode step for queries)
    c1 = batch index
    c2 = head << 16 | kv << 15 | loop << 8 | channel      (channel < 256, loop < 16)
    c3 = field << 24 | layer << 8 | sub                  (sub < 256)
"""

from dataclasses import dataclass, field
import numpy as np

from .philox import philox4x32_10

FIELD_BASE = 1
FIELD_NOISE = 2
FIELD_U = 3
FIELD_QUERY = 4
FIELD_SIGN = 5
FIELD_OUTLIER = 6

DIST_NORMAL = 0
DIST_STUDENT3 = 1

_F32 = np.float32


@dataclass(frozen=True)
class Config:
    name: str
    layers: int
    batch: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    n_loops: int
    ctx: int
    res_bits: tuple
    n_outliers: int
    outlier_mult: float
    sigma: tuple
    dist: int
    seed: int
    n_new: int = 0  # deferred-write tokens appended per sequence per step

    @property
    def group(self):
        return 32

    @property
    def gqa(self):
        return self.n_q_heads // self.n_kv_heads

    def sigma_f32(self):
        return np.array(self.sigma, dtype=_F32)


CONFIGS = (
    Config("pr1_small", 1, 1, 2, 2, 64, 4, 256, (2, 2, 2), 2, 8.0,
           (0.1, 0.1, 0.1, 0.1), DIST_NORMAL, 0),
    Config("layer_1p4b", 1, 16, 16, 16, 128, 4, 4096, (2, 2, 2), 1, 10.0,
           (0.1, 0.1, 0.1, 0.1), DIST_NORMAL, 0),
    Config("mixed_24l", 24, 64, 16, 16, 128, 4, 8192, (4, 2, 2), 1, 10.0,
           (0.2, 0.12, 0.06, 0.0), DIST_NORMAL, 0),
    Config("gqa_deep", 1, 32, 32, 8, 128, 8, 16384, (2,) * 7, 3, 16.0,
           (0.08,) * 8, DIST_STUDENT3, 0),
    Config("serving", 1, 128, 16, 16, 128, 4, 32768, (2, 2, 2), 2, 8.0,
           (0.1, 0.1, 0.1, 0.1), DIST_NORMAL, 7, n_new=1),
)


def config_by_name(name):
    for c in CONFIGS:
        if c.name == name:
            return c
    raise KeyError(name)


def _key(seed):
    return seed & 0xFFFFFFFF, (seed >> 32) & 0xFFFFFFFF


def _c2(head, kv, loop, ch):
    return ((np.asarray(head, np.uint32) << np.uint32(16))
            | (np.asarray(kv, np.uint32) << np.uint32(15))
            | (np.asarray(loop, np.uint32) << np.uint32(8))
            | np.asarray(ch, np.uint32))


def _c3(fld, layer, sub=0):
    return np.uint32((fld << 24) | ((layer & 0xFFFF) << 8) | (sub & 0xFF))


def _normal_from_words(w0, w1, w2, w3):
    """Irwin-Hall(12) normal from the twelve 10-bit fields of one Philox block."""
    s = np.zeros(np.shape(w0), dtype=np.int64)
    for w in (w0, w1, w2, w3):
        w = w.astype(np.int64)
        s += (w & 1023) + ((w >> 10) & 1023) + ((w >> 20) & 1023)
    return (s - 6138).astype(_F32) * _F32(1.0 / 1024.0)


def _normal(seed, fld, layer, sub, c0, c1, c2):
    k0, k1 = _key(seed)
    w = philox4x32_10(c0, c1, c2, _c3(fld, layer, sub), k0, k1)
    return _normal_from_words(*w)


def _student3(seed, fld, layer, c0, c1, c2):
    z0 = _normal(seed, fld, layer, 0, c0, c1, c2)
    z1 = _normal(seed, fld, layer, 1, c0, c1, c2)
    z2 = _normal(seed, fld, layer, 2, c0, c1, c2)
    z3 = _normal(seed, fld, layer, 3, c0, c1, c2)
    chi = (z1 * z1 + z2 * z2) + z3 * z3          # fp32, left to right
    v = chi / _F32(3.0)
    v = np.maximum(v, _F32(2.0 ** -10))   # bounds |t| <= 192: stays in fp16 range
    return z0 / np.sqrt(v)


def _uniform01(w):
    """(k + 0.5) / 2^24 for the top 24 bits k of a Philox word: exact in fp32."""
    k = (w >> np.uint32(8)).astype(np.int64)
    return (k.astype(_F32) + _F32(0.5)) * _F32(2.0 ** -24)


def round_bf16_f32(x):
    """Round fp32 values to the nearest bf16 (ties to even); returned as fp32."""
    x = np.ascontiguousarray(x, dtype=_F32)
    b = x.view(np.uint32).astype(np.uint64)
    lsb = (b >> np.uint64(16)) & np.uint64(1)
    r = ((b + np.uint64(0x7FFF) + lsb) >> np.uint64(16)) << np.uint64(16)
    out = r.astype(np.uint32).view(_F32)
    return np.where(np.isnan(x), x, out)


def outlier_channels(cfg, layer, head, kv):
    """The cfg.n_outliers distinct outlier channels of one (layer, kv-head, K/V)."""
    k0, k1 = _key(cfg.seed)
    chosen = []
    sub = 0
    while len(chosen) < cfg.n_outliers:
        if sub > 255:
            raise RuntimeError("outlier draw exhausted")
        w0, _, _, _ = philox4x32_10(0, 0, _c2(head, kv, 0, 0),
                                    _c3(FIELD_OUTLIER, layer, sub), k0, k1)
        ch = int(w0) % cfg.head_dim
        if ch not in chosen:
            chosen.append(ch)
        sub += 1
    return chosen


def outlier_table(cfg, layer):
    """int32 [Hkv][2][n_outliers] table of outlier channels (n_outliers may be 0)."""
    t = np.zeros((cfg.n_kv_heads, 2, max(cfg.n_outliers, 1)), dtype=np.int32) - 1
    for h in range(cfg.n_kv_heads):
        for kv in range(2):
            ch = outlier_channels(cfg, layer, h, kv)
            t[h, kv, :len(ch)] = ch
    return t


def rotation_signs(cfg, layer):
    """int8 [Hkv][2][d] Rademacher signs of the per-(layer, kv-head, K/V) rotation."""
    k0, k1 = _key(cfg.seed)
    h = np.arange(cfg.n_kv_heads)[:, None, None]
    kv = np.arange(2)[None, :, None]
    i = np.arange(cfg.head_dim)[None, None, :]
    w0, _, _, _ = philox4x32_10(0, 0, _c2(h, kv, 0, i), _c3(FIELD_SIGN, layer), k0, k1)
    return np.where((w0 & np.uint32(1)) == 0, 1, -1).astype(np.int8)


def gen_states(cfg, layer, bs, ts, heads=None, loops=None, kvs=(0, 1)):
    """bf16-valued fp32 states, shape [len(bs)][len(ts)][len(kvs)][len(loops)][len(heads)][d].

    bs, ts, heads, loops, kvs: index lists (absolute batch indices, token positions,
    kv-heads, loops, 0=K/1=V).
    """
    heads = list(range(cfg.n_kv_heads)) if heads is None else list(heads)
    loops = list(range(cfg.n_loops)) if loops is None else list(loops)
    bs = np.asarray(bs, dtype=np.int64)
    ts = np.asarray(ts, dtype=np.int64)
    d = cfg.head_dim
    k0, k1 = _key(cfg.seed)
    out = np.empty((len(bs), len(ts), len(kvs), len(loops), len(heads), d), dtype=_F32)
    sig = cfg.sigma_f32()
    ch = np.arange(d, dtype=np.uint32)
    for hi, h in enumerate(heads):
        for ki, kv in enumerate(kvs):
            mult = np.ones(d, dtype=_F32)
            for c in outlier_channels(cfg, layer, h, kv):
                mult[c] = _F32(cfg.outlier_mult)
            T0 = ts[None, :, None].astype(np.uint32)
            B0 = bs[:, None, None].astype(np.uint32)
            c2b = _c2(h, kv, 0, ch)[None, None, :]
            if cfg.dist == DIST_STUDENT3:
                base = _student3(cfg.seed, FIELD_BASE, layer, T0, B0, c2b)
            else:
                base = _normal(cfg.seed, FIELD_BASE, layer, 0, T0, B0, c2b)
            base = base * mult[None, None, :]
            for li, l in enumerate(loops):
                wu = philox4x32_10(T0[..., 0], B0[..., 0], _c2(h, kv, l, 0),
                                   _c3(FIELD_U, layer), k0, k1)[0]
                u = _F32(0.8) + _F32(0.4) * _uniform01(wu)
                n = _normal(cfg.seed, FIELD_NOISE, layer, 0, T0, B0,
                            _c2(h, kv, l, ch)[None, None, :])
                x = u[..., None] * base + sig[l] * n
                out[:, :, ki, li, hi, :] = round_bf16_f32(x)
    return out


def gen_queries(cfg, layer, bs, loops=None, step=0):
    """bf16-valued fp32 queries, shape [len(bs)][Hq][len(loops)][d]."""
    loops = list(range(cfg.n_loops)) if loops is None else list(loops)
    bs = np.asarray(bs, dtype=np.int64)
    qh = np.arange(cfg.n_q_heads, dtype=np.uint32)[None, :, None, None]
    ll = np.asarray(loops, dtype=np.uint32)[None, None, :, None]
    ch = np.arange(cfg.head_dim, dtype=np.uint32)[None, None, None, :]
    B0 = bs.astype(np.uint32)[:, None, None, None]
    z = _normal(cfg.seed, FIELD_QUERY, layer, 0, np.uint32(step), B0, _c2(qh, 0, ll, ch))
    return round_bf16_f32(z)
