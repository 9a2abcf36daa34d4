"""Parity between librq (GPU) and the fp64 oracle on the same seeded inputs.

Encode parity is conditional (GPU arithmetic is fp32, the oracle's fp64): for every stored
fp16 value (step, offset, a_l) and every code, the oracle recomputes the value; where the
GPU's value differs, it is accepted only if the two are neighbours and the oracle's
pre-rounding value lies within 1e-6 (relative to the value for fp16 quantities, in code
units for codes) of the boundary between them.  The oracle then continues with the GPU's
choice.  Everything else must match bit for bit, packed bytes included.  Reported counts:
codes whose value lies within the band (`band`, out of `codes`; exact half-way ties, which
both sides round to even, included) and elements where the GPU's neighbouring choice was
taken (`followed`, out of `elements`), which must stay below 1e-5 of all elements.

Output parity: GPU bf16 output vs the oracle's fp64 output,
    max over elements of (|gpu - ref| - ulp_bf16(ref)/2) <= 2e-3,
    mean over elements of max(0, |gpu - ref| - ulp_bf16(ref)/2) <= 2e-4,
i.e. the error budget is for the arithmetic, on top of the unavoidable rounding of the
result to bf16.
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
        self.band = 0          # codes whose pre-rounding value lies within the band
        self.followed = 0      # elements where the GPU's neighbouring choice was taken
        self.bad = 0           # any other disagreement
        self.bad_names = {}

    def __call__(self, name, pre, rounded):
        g = np.asarray(self.gpu[name], dtype=np.float64).reshape(np.shape(rounded))
        pre = np.asarray(pre, dtype=np.float64)
        rounded = np.asarray(rounded, dtype=np.float64)
        diff = g != rounded
        if name.endswith("_c"):
            band = np.abs(pre - (np.floor(pre) + 0.5)) <= CODE_BAND
            near = diff & (np.abs(g - rounded) == 1) & \
                (np.abs(pre - (g + rounded) / 2) <= CODE_BAND)
            self.codes += rounded.size
            self.band += int(band.sum())
        else:
            toward = np.where(g > rounded, np.float16(np.inf), np.float16(-np.inf))
            adjacent = np.nextafter(rounded.astype(np.float16),
                                    toward.astype(np.float16)).astype(np.float64) == g
            near = diff & adjacent & (np.abs(pre - (g + rounded) / 2) <= REL_BAND * np.abs(pre))
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
    return {"max_excess": float(excess.max(initial=0.0)), "mean_excess": float(excess.mean()),
            "max_abs": float(err.max(initial=0.0)), "mean_abs": float(err.mean())}


def check_slice(w, b, h, loop_calls, outs, pending=True, check_encode=True):
    """Encode parity and output parity for sequence b, kv-head h of workload w.

    loop_calls: list of (loop_begin, loop_count); outs: matching GPU outputs (torch bf16
    [B][Hq][loop_count][d]).  Returns a stats dict; raises AssertionError on a failure.
    """
    cfg, d, L = w.cfg, w.d, w.L
    res_bits = list(cfg.res_bits[: L - 1])
    ctx = w.ctx_list[b]
    ntok = max(ctx, 1)
    ntok_e = ntok + ntok % 2
    x = synth.gen_states(cfg, w.layer, [b], np.arange(ntok_e), heads=[h])[0, :, :, :, 0, :]
    x = x.astype(np.float64)                                      # [ntok][2][L][d]
    sl = w.packed_slice(b, h, ntok_e)
    signs = w.signs_np[h].astype(np.float64)                      # [2][d]
    stats = {"elements": 0, "codes": 0, "band": 0, "followed": 0}
    encs = []
    for kv in range(2):
        f = Follow(gpu_slice_to_oracle_names(sl, kv, d, L, res_bits))
        enc = O.encode(x[:, kv], signs[kv], res_bits, rnd=f)
        assert f.bad == 0, "encode mismatch kv=%d b=%d h=%d: %s" % (kv, b, h, f.bad_names)
        if check_encode:
            assert packed_bytes_equal(enc, sl, kv, res_bits), "packed bytes differ kv=%d" % kv
        stats["elements"] += f.total
        stats["codes"] += f.codes
        stats["band"] += f.band
        stats["followed"] += f.followed
        encs.append(enc_head(enc, ctx))
    pend = synth.gen_states(cfg, w.layer, [b], [ctx], heads=[h])[0, 0, :, :, 0, :] \
        .astype(np.float64) if pending else None                  # [2][L][d]
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
    assert stats["max_excess"] <= MAX_ABS, stats
    assert stats["mean_excess"] <= MEAN_ABS, stats
    return stats
