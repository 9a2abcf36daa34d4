"""Parity between librq (GPU) and the fp64 oracle on the same seeded inputs.

Encode parity is conditional (GPU arithmetic is fp32, the oracle's fp64): for every stored
fp16 value (step, offset, a_l) and every code, the oracle recomputes the value; where the
GPU's value differs, it is accepted only if the two are neighbours and the oracle's
pre-rounding value lies within 1e-6 of the rounding boundary between them (relative to the
value for fp16 quantities; relative to the spacing of the boundaries, i.e. in code units,
for codes).  The oracle then continues with the GPU's choice.  Everything else must match
bit for bit, packed bytes included.

Counted separately for packed codes and for fp16 values:
  ties       the fp64 pre-rounding value lies exactly on a boundary (a code quotient of
             k + 1/2, an fp16 midpoint): both sides round it to even, so it cannot differ;
  near       the value lies within the band but not exactly on the boundary: the elements
             where fp32 and fp64 arithmetic could take different neighbours;
  followed   elements where the GPU did take the other neighbour.
The near-boundary criterion is on packed codes: code `near` < 1e-5 of all codes.  For fp16
values the band (1e-6 relative around midpoints 2^-10 relative apart) holds about 0.2% of any
generic quantity whatever computes it, so there the bound is on the choices actually taken:
`followed` (codes and fp16 values) < 1e-5 of all elements.

Output parity: GPU bf16 output vs the oracle's fp64 output,
    max over elements of (|gpu - ref| - ulp_bf16(ref)/2) <= 2e-3,
    mean over elements of max(0, |gpu - ref| - ulp_bf16(ref)/2) <= 2e-4,
i.e. the error budget is for the arithmetic, on top of the unavoidable rounding of the
result to bf16.  Also reported: the fraction of outputs not equal to bf16_rne(ref) and the
fraction more than one bf16 ulp away from it.
"""

import numpy as np

import oracle as O
import synth

REL_BAND = 1e-6
CODE_BAND = 1e-6
MAX_ABS = 2e-3
MEAN_ABS = 2e-4


def _fp16_neighbour_mid(pre, rounded):
    """Midpoint between `rounded` and its fp16 neighbour on the side of `pre`."""
    h = rounded.astype(np.float16)
    toward = np.where(pre >= rounded, np.float16(np.inf), np.float16(-np.inf)).astype(np.float16)
    other = np.nextafter(h, toward).astype(np.float64)
    return (rounded + other) / 2


class Follow:
    def __init__(self, gpu):
        self.gpu = gpu
        self.total = 0
        self.codes = 0         # packed codes checked
        self.ties = 0          # codes: pre-rounding quotient exactly k + 1/2 (both round to even)
        self.near = 0          # codes: within the band, not exactly on the boundary
        self.f16_ties = 0      # fp16 values exactly on a midpoint
        self.f16_near = 0      # fp16 values within the band, not on the midpoint
        self.followed = 0      # elements where the GPU's neighbouring choice was taken
        self.bad = 0           # any other disagreement
        self.bad_names = {}

    def __call__(self, name, pre, rounded):
        g = np.asarray(self.gpu[name], dtype=np.float64).reshape(np.shape(rounded))
        pre = np.asarray(pre, dtype=np.float64)
        rounded = np.asarray(rounded, dtype=np.float64)
        diff = g != rounded
        if name.endswith("_c"):
            dist = np.abs(pre - (np.floor(pre) + 0.5))      # to the nearest boundary
            in_band = dist <= CODE_BAND
            near = diff & (np.abs(g - rounded) == 1) & \
                (np.abs(pre - (g + rounded) / 2) <= CODE_BAND)
            self.codes += rounded.size
            self.ties += int((in_band & (dist == 0)).sum())
            self.near += int((in_band & (dist > 0)).sum())
        else:
            dist = np.abs(pre - _fp16_neighbour_mid(pre, rounded))   # boundary on pre's side
            in_band = dist <= REL_BAND * np.abs(pre)
            toward = np.where(g > rounded, np.float16(np.inf), np.float16(-np.inf))
            adjacent = np.nextafter(rounded.astype(np.float16),
                                    toward.astype(np.float16)).astype(np.float64) == g
            near = diff & adjacent & (np.abs(pre - (g + rounded) / 2) <= REL_BAND * np.abs(pre))
            self.f16_ties += int((in_band & (dist == 0)).sum())
            self.f16_near += int((in_band & (dist > 0)).sum())
        bad = diff & ~near
        self.total += rounded.size
        self.followed += int(near.sum())
        nb = int(bad.sum())
        if nb:
            self.bad += nb
            self.bad_names[name] = self.bad_names.get(name, 0) + nb
        return np.where(near, g, rounded)


def gpu_slice_to_oracle_names(sl, kv, d, L, res_bits):
    """Map packed arrays of one (b, h) slice to the oracle's rounding-hook names."""
    n = sl[("ref_codes", kv)].shape[0]

    def natural(stored, bits):
        if kv == 1:
            return O.v_unlayout(stored.reshape(n // 2, -1), stored.shape[1])
        return O.k_unlayout(stored, bits, d)

    rows = natural(sl[("ref_codes", kv)], 4)
    out = {"ref_c": O.unpack_rows(rows, 4, d), "ref_s": sl[("ref_meta", kv)][..., 0],
           "ref_z": sl[("ref_meta", kv)][..., 1]}
    for l in range(L - 1):
        rows = natural(sl[("res_codes", kv, l)], res_bits[l])
        out["res%d_c" % l] = O.unpack_rows(rows, res_bits[l], d)
        out["res%d_s" % l] = sl[("res_meta", kv, l)][..., 0]
        out["res%d_z" % l] = sl[("res_meta", kv, l)][..., 1]
        out["alpha%d" % l] = sl[("alpha", kv, l)]
    return out


def packed_bytes_equal(enc, sl, kv, res_bits):
    """The oracle's own packing of its (followed) codes equals the GPU's bytes."""
    n = sl[("ref_codes", kv)].shape[0]
    d = enc["ref"][0].shape[1]

    def lay(rows, bits):
        return O.v_layout(rows).reshape(n, -1) if kv == 1 else O.k_layout(rows, bits, d)

    ok = np.array_equal(lay(O.pack_rows(enc["ref"][0], 4), 4), sl[("ref_codes", kv)])
    for l, (c, s, z) in enumerate(enc["res"]):
        ok &= np.array_equal(lay(O.pack_rows(c, res_bits[l]), res_bits[l]),
                             sl[("res_codes", kv, l)])
        ok &= np.array_equal(s, sl[("res_meta", kv, l)][..., 0])
        ok &= np.array_equal(z, sl[("res_meta", kv, l)][..., 1])
        ok &= np.array_equal(enc["alpha"][l], sl[("alpha", kv, l)])
    ok &= np.array_equal(enc["ref"][1], sl[("ref_meta", kv)][..., 0])
    ok &= np.array_equal(enc["ref"][2], sl[("ref_meta", kv)][..., 1])
    return bool(ok)


def enc_head(enc, n):
    if n == 0:
        return None
    return {"ref": tuple(a[:n] for a in enc["ref"]),
            "alpha": [a[:n] for a in enc["alpha"]],
            "res": [tuple(a[:n] for a in r) for r in enc["res"]]}


def bf16_half_ulp(x):
    ax = np.abs(np.asarray(x, dtype=np.float64))
    e = np.floor(np.log2(np.where(ax > 0, ax, 1.0)))
    return np.where(ax > 0, np.ldexp(1.0, (e - 8).astype(int)), 0.0)


def output_errors(gpu, ref):
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    err = np.abs(gpu - ref)
    excess = np.maximum(err - bf16_half_ulp(ref), 0.0)
    # against the correctly rounded result: bf16_rne(ref) and one bf16 ulp at its magnitude
    rne = O.bf16_round(ref)
    ulp = 2.0 * bf16_half_ulp(rne)
    off = np.abs(gpu - rne)
    return {"max_excess": float(excess.max(initial=0.0)), "mean_excess": float(excess.mean()),
            "max_abs": float(err.max(initial=0.0)), "mean_abs": float(err.mean()),
            "n": int(gpu.size), "not_rne": int(np.count_nonzero(off)),
            "beyond_1ulp": int(np.count_nonzero(off > ulp))}


def check_slice(w, b, h, loop_calls, outs, pending=True, check_encode=True, cache=None,
                states=None, ctx=None, pending_state=None, encode=None):
    """Encode parity and output parity for sequence b, kv-head h of workload w.

    loop_calls: list of (loop_begin, loop_count); outs: matching GPU outputs (torch bf16
    [B][Hq][loop_count][d]).  By default the slice's tokens are the generator's states at
    positions 0..ctx-1 (ctx = w.ctx_list[b]) and the current token is the generator's state at
    position ctx.  A caller whose cache holds other tokens (a serving run that appended
    tokens) passes them: states [n][2][L][d] (n >= ctx: every stored token to check, the
    first ctx of them attended), ctx, and pending_state [2][L][d].  cache: a paged twin
    (PackedCache with n_pages) whose pages hold the slice, read through w's block table
    argument instead of w's contiguous cache (cache=(paged_cache, table_numpy)).  encode: the
    oracle encode to follow (default oracle.encode; an ablation passes its own variant).
    Returns a stats dict; raises AssertionError on a failure.
    """
    cfg, d, L = w.cfg, w.d, w.L
    res_bits = list(cfg.res_bits[: L - 1])
    ctx = w.ctx_list[b] if ctx is None else ctx
    if states is None:
        ntok = max(ctx, 1)
        ntok_e = ntok + ntok % 2
        x = synth.gen_states(cfg, w.layer, [b], np.arange(ntok_e), heads=[h])[0, :, :, :, 0, :]
    else:
        x = np.asarray(states)
        ntok_e = x.shape[0]
        assert ntok_e % 2 == 0 and ntok_e >= ctx
    x = x.astype(np.float64)                                      # [ntok][2][L][d]
    if cache is None:
        sl = w.packed_slice(b, h, ntok_e)
    else:
        sl = w.packed_slice_paged(cache[0], cache[1], b, h, ntok_e)
    signs = w.signs_np[h].astype(np.float64)                      # [2][d]
    stats = {"elements": 0, "codes": 0, "ties": 0, "near": 0, "f16_ties": 0, "f16_near": 0,
             "followed": 0}
    encs = []
    for kv in range(2):
        f = Follow(gpu_slice_to_oracle_names(sl, kv, d, L, res_bits))
        enc = (encode or O.encode)(x[:, kv], signs[kv], res_bits, rnd=f)
        assert f.bad == 0, "encode mismatch kv=%d b=%d h=%d: %s" % (kv, b, h, f.bad_names)
        if check_encode:
            assert packed_bytes_equal(enc, sl, kv, res_bits), "packed bytes differ kv=%d" % kv
        stats["elements"] += f.total
        stats["codes"] += f.codes
        stats["ties"] += f.ties
        stats["near"] += f.near
        stats["f16_ties"] += f.f16_ties
        stats["f16_near"] += f.f16_near
        stats["followed"] += f.followed
        encs.append(enc_head(enc, ctx))
    if not pending:
        pend = None
    elif pending_state is not None:
        pend = np.asarray(pending_state, np.float64)              # [2][L][d]
    else:
        pend = synth.gen_states(cfg, w.layer, [b], [ctx], heads=[h])[0, 0, :, :, 0, :] \
            .astype(np.float64)
    qall = synth.gen_queries(cfg, w.layer, [b])[0].astype(np.float64)   # [Hq][L][d]
    g = w.Hq // w.H
    errs = []
    for (l0, lc), out in zip(loop_calls, outs):
        got = out[b, h * g:(h + 1) * g].float().cpu().numpy().astype(np.float64)  # [g][lc][d]
        for li in range(lc):
            l = l0 + li
            q = qall[h * g:(h + 1) * g, l]
            if ctx == 0 and not pending:
                ref = np.zeros((g, d))
            else:
                ref = O.decode_rotated(q, encs[0], encs[1], signs[0], signs[1], l,
                                       pend[0, l] if pending else None,
                                       pend[1, l] if pending else None)
            errs.append(output_errors(got[:, li], ref))
    stats["max_excess"] = max(e["max_excess"] for e in errs)
    stats["mean_excess"] = float(np.mean([e["mean_excess"] for e in errs]))
    stats["max_abs"] = max(e["max_abs"] for e in errs)
    stats["mean_abs"] = float(np.mean([e["mean_abs"] for e in errs]))
    stats["outputs"] = sum(e["n"] for e in errs)
    stats["not_rne"] = sum(e["not_rne"] for e in errs)
    stats["beyond_1ulp"] = sum(e["beyond_1ulp"] for e in errs)
    assert stats["max_excess"] <= MAX_ABS, stats
    assert stats["mean_excess"] <= MEAN_ABS, stats
    return stats
