"""Plain fp64 CPU oracle of ResidualQuant encode and decode attention.

TEST INFRASTRUCTURE ONLY.  Only the test suite, the package's smoke check and the
benchmark's CPU-baseline leg may import this module.  The product path (the native
library and its Python binding) never calls it, and this module imports nothing from
the product package.

Sources (the two pages that describe the method):
  [A] "ResidualQuant: KV Cache Quantization for Looped Transformers with 2-Bit
      Residuals", abstract (final-loop reference, low-precision residuals,
      least-squares scaling, rotations of the residuals, loop-wise mixed precision).
  [B] the rit.work summary "ResidualQuant: KV cache of looped transformers", sections
      "How each pass's KV cache is reconstructed" (final-pass reference, LS scale per
      difference, rotation in channel space calibrated per layer/head/K-V, INT4
      reference and INT2 residuals with an adjustable step and offset that use every
      level, deferred write of the current token in BF16, fused kernel that rebuilds
      reference and residuals inside attention).

Readings where the pages are silent (each restated where it is used):
  * groups of 32 contiguous channels; the reference is grouped in the original basis,
    residuals in the rotated basis;
  * step s = (max - min) / (2^b - 1), offset z = min, both stored as fp16 (RNE); codes
    are round-half-even of (x - z_h) / s_h clamped to [0, 2^b - 1]; a group whose
    stored step is 0 gets codes 0 and dequantises to z_h;
  * one LS scale a per (token, kv-head, loop, K/V), stored fp16; a = 0 when the
    dequantised reference is all zero; the residual uses the stored a_h and the
    dequantised reference, so decode rebuilds exactly what encode quantised;
  * R = H_d diag(signs) / sqrt(d) with the Sylvester Hadamard H_d and per
    (layer, kv-head, K/V) random signs, standing in for the calibrated rotation;
  * softmax scale 1/sqrt(d); query head h reads kv-head h // (Hq / Hkv); a loop-l query
    attends over loop l's reconstructed cache plus the current token's BF16 K/V.

Every rounding step goes through a `rnd` hook: by default it returns round-to-nearest-
even; a parity test may pass a hook that compares with another implementation's
stored value and follows that value where the pre-rounding quantity lies within the
accepted distance of a rounding boundary.
"""

import numpy as np
import scipy.linalg

GROUP = 32


# ----------------------------------------------------------------------------- rounding

def fp16_round(x):
    """Nearest fp16 value (ties to even), returned as fp64."""
    return np.asarray(x, dtype=np.float64).astype(np.float16).astype(np.float64)


def bf16_round(x):
    """Nearest bf16 value (8 significant bits, ties to even), returned as fp64.

    Written directly on the fp64 value (frexp / rint / ldexp) so that no intermediate
    fp32 rounding happens.  Finite inputs only.
    """
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)                    # x = m * 2^e, 0.5 <= |m| < 1
    e = np.maximum(e, -125)               # bf16 subnormals share fp32's exponent floor
    return np.ldexp(np.rint(np.ldexp(x, 8 - e)), e - 8)


def default_rnd(name, pre, rounded):
    return rounded


# ------------------------------------------------------------------------- quantisation

def group_view(v):
    """[..., d] -> [..., d/32, 32] view of contiguous channel groups."""
    v = np.asarray(v, dtype=np.float64)
    return v.reshape(v.shape[:-1] + (v.shape[-1] // GROUP, GROUP))


def step_offset(v, bits):
    """Asymmetric min/max quantiser of [B]: s = (max - min)/(2^b - 1), z = min, per group.

    Returns the pre-rounding (s, z) in fp64, shape [..., d/32].
    """
    g = group_view(v)
    mn = g.min(axis=-1)
    mx = g.max(axis=-1)
    return (mx - mn) / (2 ** bits - 1), mn


def code_quotient(v, s_h, z_h):
    """(v - z_h) / s_h per element (0 where s_h == 0), shape [..., d]."""
    g = group_view(v)
    s = s_h[..., None]
    with np.errstate(divide="ignore", invalid="ignore"):
        q = np.where(s > 0, (g - z_h[..., None]) / np.where(s > 0, s, 1.0), 0.0)
    return q.reshape(np.shape(v))


def codes_from_quotient(q, bits):
    return np.clip(np.rint(q), 0, 2 ** bits - 1)


def dequant(c, s_h, z_h):
    """c * s_h + z_h per group, shape [..., d]."""
    g = group_view(c)
    return (g * s_h[..., None] + z_h[..., None]).reshape(np.shape(c))


def quantize(v, bits, tag, rnd=default_rnd):
    """Group-quantise v [..., d] to `bits` bits; returns (codes, s_h, z_h) as fp64 arrays."""
    s, z = step_offset(v, bits)
    s_h = rnd(tag + "_s", s, fp16_round(s))
    z_h = rnd(tag + "_z", z, fp16_round(z))
    q = code_quotient(v, s_h, z_h)
    c = rnd(tag + "_c", q, codes_from_quotient(q, bits))
    return c, s_h, z_h


# ---------------------------------------------------------------------- LS scale, rotation

def ls_scale(x, ref_hat):
    """a = <x, ref_hat> / <ref_hat, ref_hat>: the minimiser of ||x - a ref_hat|| ([A], [B]).

    0 where the dequantised reference is all zero.  Shape [...] for inputs [..., d].
    """
    x = np.asarray(x, dtype=np.float64)
    r = np.asarray(ref_hat, dtype=np.float64)
    num = np.sum(x * r, axis=-1)
    den = np.sum(r * r, axis=-1)
    with np.errstate(divide="ignore", invalid="ignore"):
        return np.where(den > 0, num / np.where(den > 0, den, 1.0), 0.0)


def hadamard(d):
    """Sylvester Hadamard matrix H_d (entries +-1, symmetric, H H = d I)."""
    return scipy.linalg.hadamard(d).astype(np.float64)


def rotation(signs):
    """R = H_d diag(signs) / sqrt(d): orthogonal, one per (layer, kv-head, K/V) ([B])."""
    s = np.asarray(signs, dtype=np.float64)
    d = s.shape[-1]
    return hadamard(d) * s[None, :] / np.sqrt(d)


# ------------------------------------------------------------------------------ encode

def encode(x, signs, res_bits, rnd=default_rnd):
    """Encode the loop states of tokens after the final loop has finished ([B], deferred write).

    x:        [N][L][d] fp64 (the bf16 states of N token-heads of one K or V)
    signs:    [d] rotation signs of this (layer, kv-head, K/V)
    res_bits: residual bit width of each non-final loop (length L-1)

    Returns a dict with, per token, the INT4 reference (codes, s, z), and per non-final
    loop l the LS scale a_l and the rotated residual's (codes, s, z).
    """
    x = np.asarray(x, dtype=np.float64)
    L = x.shape[1]
    R = rotation(signs)
    # reference: the final loop's state, INT4 ([A], [B])
    rc, rs, rz = quantize(x[:, L - 1, :], 4, "ref", rnd)
    ref_hat = dequant(rc, rs, rz)
    out = {"ref": (rc, rs, rz), "alpha": [], "res": []}
    for l in range(L - 1):
        # least-squares scale of loop l against the dequantised reference ([A], [B])
        a = ls_scale(x[:, l, :], ref_hat)
        a_h = rnd("alpha%d" % l, a, fp16_round(a))
        # residual against the scaled reference, then the channel rotation ([B])
        r = x[:, l, :] - a_h[:, None] * ref_hat
        y = r @ R.T
        c, s, z = quantize(y, res_bits[l], "res%d" % l, rnd)
        out["alpha"].append(a_h)
        out["res"].append((c, s, z))
    return out


def reconstruct(enc, signs):
    """K_l = a_l * deq4(ref) + R^T deq(res_l) for l < L-1; K_{L-1} = deq4(ref).  [N][L][d]."""
    R = rotation(signs)
    rc, rs, rz = enc["ref"]
    ref_hat = dequant(rc, rs, rz)
    loops = []
    for l, (c, s, z) in enumerate(enc["res"]):
        e = dequant(c, s, z)
        loops.append(enc["alpha"][l][:, None] * ref_hat + e @ R)
    loops.append(ref_hat)
    return np.stack(loops, axis=1)


# -------------------------------------------------------------------------- attention

def softmax_attention(q, K, V, scale):
    """Textbook softmax(q K^T * scale) V in fp64.  q [M][d], K/V [T][d] -> [M][d]."""
    s = (np.asarray(q, np.float64) @ np.asarray(K, np.float64).T) * scale
    s = s - s.max(axis=-1, keepdims=True)
    p = np.exp(s)
    p = p / p.sum(axis=-1, keepdims=True)
    return p @ np.asarray(V, np.float64)


def decode_explicit(q, enc_k, enc_v, signs_k, signs_v, loop, pending_k=None,
                    pending_v=None, scale=None):
    """Form (a): rebuild loop `loop`'s K/V explicitly and run textbook attention.

    q: [M][d] queries of loop `loop` for the query heads of one kv-head.
    enc_k / enc_v: encode() results for the ctx tokens of that kv-head.
    pending_k/v: [d] the current token's BF16 state of this loop, or None ([B]).
    """
    q = np.asarray(q, np.float64)
    d = q.shape[-1]
    scale = 1.0 / np.sqrt(d) if scale is None else scale
    K = reconstruct(enc_k, signs_k)[:, loop, :] if enc_k is not None else np.zeros((0, d))
    V = reconstruct(enc_v, signs_v)[:, loop, :] if enc_v is not None else np.zeros((0, d))
    if pending_k is not None:
        K = np.concatenate([K, np.asarray(pending_k, np.float64)[None, :]], axis=0)
        V = np.concatenate([V, np.asarray(pending_v, np.float64)[None, :]], axis=0)
    return softmax_attention(q, K, V, scale)


def decode_rotated(q, enc_k, enc_v, signs_k, signs_v, loop, pending_k=None,
                   pending_v=None, scale=None):
    """Form (b): the same attention with the rotation moved onto the query and the output.

    score_t = a_t (q . ref_hat_t) + (R q) . e_t;  out = (sum_t p_t a_t ref_hat_t
    + R^T sum_t p_t e_t + p_pend v_pend) / sum p, where e_t is the dequantised rotated
    residual ([B]: the kernel rebuilds reference and residual inside attention and never
    writes the decompressed K/V back).  Equals form (a) up to fp64 rounding.
    """
    q = np.asarray(q, np.float64)
    M, d = q.shape
    scale = 1.0 / np.sqrt(d) if scale is None else scale
    Rk = rotation(signs_k)
    Rv = rotation(signs_v)
    L = len(enc_k["res"]) + 1 if enc_k is not None else loop + 1
    scores = []
    terms_ref = []
    terms_res = []
    if enc_k is not None:
        kref = dequant(*enc_k["ref"])
        vref = dequant(*enc_v["ref"])
        if loop < L - 1:
            ak = enc_k["alpha"][loop]
            av = enc_v["alpha"][loop]
            ek = dequant(*enc_k["res"][loop])
            ev = dequant(*enc_v["res"][loop])
            qr = q @ Rk.T                                 # q' = R q
            s = (ak[None, :] * (q @ kref.T) + qr @ ek.T) * scale
            terms_ref.append((av[:, None] * vref))
            terms_res.append(ev)
        else:
            s = (q @ kref.T) * scale
            terms_ref.append(vref)
            terms_res.append(np.zeros_like(vref))
        scores.append(s)
    if pending_k is not None:
        scores.append((q @ np.asarray(pending_k, np.float64))[:, None] * scale)
        terms_ref.append(np.asarray(pending_v, np.float64)[None, :])
        terms_res.append(np.zeros((1, d)))
    s = np.concatenate(scores, axis=1)
    m = s.max(axis=1, keepdims=True)
    p = np.exp(s - m)
    ell = p.sum(axis=1, keepdims=True)
    acc_ref = p @ np.concatenate(terms_ref, axis=0)
    acc_res = p @ np.concatenate(terms_res, axis=0)
    return (acc_ref + acc_res @ Rv) / ell


# ----------------------------------------------------------------------------- packing

def pack_rows(codes, bits):
    """Pack codes [N][d] of `bits` bits little-endian: channel i sits in byte i*bits//8 at
    bit offset (i*bits) % 8.  Returns uint8 [N][d*bits/8]."""
    c = np.asarray(codes).astype(np.uint32)
    N, d = c.shape
    per = 8 // bits
    c = c.reshape(N, d // per, per)
    out = np.zeros((N, d // per), dtype=np.uint32)
    for j in range(per):
        out |= c[:, :, j] << np.uint32(bits * j)
    return out.astype(np.uint8)


def unpack_rows(rows, bits, d):
    r = np.asarray(rows, dtype=np.uint8).astype(np.uint32)
    per = 8 // bits
    mask = np.uint32(2 ** bits - 1)
    out = np.stack([(r >> np.uint32(bits * j)) & mask for j in range(per)], axis=-1)
    return out.reshape(r.shape[0], d).astype(np.float64)


def k_word_order(d, bits):
    """Physical 32-bit word of each natural word of a K code row.

    A K row stores its words group-interleaved: natural word w (channels of group w // bits,
    k-th word of that group, k = w % bits) sits at word k * (d/32) + w // bits, so the k-th
    words of all groups are adjacent."""
    ng = d // GROUP
    w = np.arange(d * bits // 32)
    return (w % bits) * ng + w // bits


def k_layout(rows, bits, d):
    """Natural code rows [N][d*bits/8] -> the bytes stored for K rows."""
    r = np.asarray(rows, dtype=np.uint8)
    N, rb = r.shape
    words = r.reshape(N, rb // 4, 4)
    out = np.empty_like(words)
    out[:, k_word_order(d, bits), :] = words
    return out.reshape(N, rb)


def k_unlayout(stored, bits, d):
    r = np.asarray(stored, dtype=np.uint8)
    N, rb = r.shape
    return r.reshape(N, rb // 4, 4)[:, k_word_order(d, bits), :].reshape(N, rb)


def v_unit_swizzle(p, units):
    """XOR applied to the 16-bit unit index u in the row pair p of a V code array: 8 (p mod 4)
    for 32-unit rows, 8 ((p div 2) mod 2) for 16-unit rows, none for shorter rows."""
    p = np.asarray(p)
    if units == 32:
        return 8 * (p & 3)
    if units == 16:
        return 8 * ((p >> 1) & 1)
    return np.zeros_like(p)


def v_layout(rows):
    """V-side token-pair layout of natural code rows [N][rb] (N even, rb even) -> [N/2][2*rb]:
    in pair p (tokens 2p, 2p+1) the 32-bit word at position u ^ swizzle(p) holds 16-bit unit u
    of token 2p (low half) and of token 2p+1 (high half)."""
    r = np.asarray(rows, dtype=np.uint8)
    N, rb = r.shape
    units = rb // 2
    u = r.reshape(N // 2, 2, units, 2)                      # [pair][tok][unit][byte]
    pairs = np.ascontiguousarray(u.transpose(0, 2, 1, 3))   # [pair][unit][tok][byte]
    out = np.empty_like(pairs)
    for p in range(N // 2):
        pos = np.arange(units) ^ v_unit_swizzle(p, units)
        out[p, pos] = pairs[p]
    return out.reshape(N // 2, 2 * rb)


def v_unlayout(stored, rb):
    s = np.asarray(stored, dtype=np.uint8)
    P = s.shape[0]
    units = rb // 2
    w = s.reshape(P, units, 2, 2)
    pairs = np.empty_like(w)
    for p in range(P):
        pos = np.arange(units) ^ v_unit_swizzle(p, units)
        pairs[p] = w[p, pos]
    return np.ascontiguousarray(pairs.transpose(0, 2, 1, 3)).reshape(2 * P, rb)


def cache_bytes(d, n_loops, res_bits, tokens, heads=1, batch=1):
    """Bytes of the packed cache (K and V): per token-head, the reference (d/2 code bytes
    + 4 bytes of fp16 step/offset per group) plus, per non-final loop l, d*b_l/8 code bytes,
    4 bytes per group and 2 bytes of fp16 a_l."""
    ng = d // GROUP
    per = d // 2 + 4 * ng
    for b in res_bits[: n_loops - 1]:
        per += d * b // 8 + 4 * ng + 2
    return 2 * per * tokens * heads * batch
