"""Ablation variants of the encode, built from the fp64 oracle's steps (test infrastructure).

Each variant drops or changes one step of the method ("ResidualQuant: KV Cache Quantization
for Looped Transformers with 2-Bit Residuals", abstract: direct INT2 quantisation of the loops
fails, the LS scale and the rotation each reduce the error; rit.work summary, "How each
pass's KV cache is reconstructed"):
  rq           the method: INT4 final-loop reference, LS scale a_l, rotated residual
  direct       every non-final loop quantised directly at its residual bit width, no reference
  direct_rotated  the same in the rotated basis (what the GPU ablation kernel decodes)
  no_ls        a_l = 1 (residual against the unscaled reference)
  no_rotation  R = I (residual quantised in original channels)
  chained      loop l's reference is the reconstruction of loop l + 1 (a chain towards the
               final loop) instead of the final loop itself
The final loop is the INT4 reference in every variant.  All functions take the states of
one K or V, x [N][L][d], and return the reconstruction [N][L][d].
"""

import numpy as np

import oracle as O


def recon_rq(x, signs, res_bits):
    return O.reconstruct(O.encode(x, signs, res_bits), signs)


def _ref_hat(x):
    L = x.shape[1]
    return O.dequant(*O.quantize(x[:, L - 1, :], 4, "ref"))


def recon_direct(x, signs, res_bits):
    L = x.shape[1]
    out = [O.dequant(*O.quantize(x[:, l, :], res_bits[l], "d%d" % l)) for l in range(L - 1)]
    out.append(_ref_hat(x))
    return np.stack(out, axis=1)


def _residual_loops(x, signs, res_bits, scale, rotate, chain):
    L = x.shape[1]
    R = O.rotation(signs) if rotate else np.eye(x.shape[2])
    ref_hat = _ref_hat(x)
    out = [None] * L
    out[L - 1] = ref_hat
    for l in range(L - 2, -1, -1):
        base = out[l + 1] if chain else ref_hat
        a = O.fp16_round(O.ls_scale(x[:, l, :], base)) if scale else np.ones(x.shape[0])
        r = x[:, l, :] - a[:, None] * base
        c, s, z = O.quantize(r @ R.T, res_bits[l], "r%d" % l)
        out[l] = a[:, None] * base + O.dequant(c, s, z) @ R
    return np.stack(out, axis=1)


def recon_no_ls(x, signs, res_bits):
    return _residual_loops(x, signs, res_bits, scale=False, rotate=True, chain=False)


def recon_no_rotation(x, signs, res_bits):
    return _residual_loops(x, signs, res_bits, scale=True, rotate=False, chain=False)


def recon_chained(x, signs, res_bits):
    return _residual_loops(x, signs, res_bits, scale=True, rotate=True, chain=True)


def encode_fixed_alpha(x, signs, res_bits, a_value, rnd=O.default_rnd):
    """The oracle's encode steps with the LS scale replaced by a fixed a (1: residual against
    the unscaled reference; 0: the loop's own state rotated and quantised directly), with the
    same rounding hook as oracle.encode so that a GPU encode can be followed code for code."""
    x = np.asarray(x, dtype=np.float64)
    L = x.shape[1]
    R = O.rotation(signs)
    rc, rs, rz = O.quantize(x[:, L - 1, :], 4, "ref", rnd)
    ref_hat = O.dequant(rc, rs, rz)
    out = {"ref": (rc, rs, rz), "alpha": [], "res": []}
    for l in range(L - 1):
        a = np.full(x.shape[0], float(a_value))            # exact in fp16
        a_h = rnd("alpha%d" % l, a, a)
        y = (x[:, l, :] - a_h[:, None] * ref_hat) @ R.T
        c, s, z = O.quantize(y, res_bits[l], "res%d" % l, rnd)
        out["alpha"].append(a_h)
        out["res"].append((c, s, z))
    return out


def recon_direct_rotated(x, signs, res_bits):
    """Direct quantisation of every non-final loop in the rotated basis (a = 0): the format the
    GPU ablation kernel decodes; the rotation costs the decode nothing (one transform of the
    query and one of the accumulator), so its bytes and time are those of direct INT2."""
    return O.reconstruct(encode_fixed_alpha(x, signs, res_bits, 0.0), signs)


VARIANTS = {"rq": recon_rq, "direct": recon_direct, "direct_rotated": recon_direct_rotated,
            "no_ls": recon_no_ls, "no_rotation": recon_no_rotation, "chained": recon_chained}


def bytes_per_token_head(variant, d, res_bits):
    """Stored bytes per token-head (K and V) of a variant's cache."""
    ng = d // 32
    per = d // 2 + 4 * ng                                   # INT4 reference + its meta
    for b in res_bits:
        per += d * b // 8 + 4 * ng + (0 if variant in ("direct", "direct_rotated", "no_ls") else 2)
    return 2 * per


def rel_err(x, xh):
    """||x - xh|| / ||x|| per loop (over tokens and channels): [L]."""
    return np.sqrt(((x - xh) ** 2).sum(axis=(0, 2)) / (x ** 2).sum(axis=(0, 2)))


def attention_rel_err(q, K, V, Kh, Vh, scale):
    """Per loop: ||attn(q, Kh, Vh) - attn(q, K, V)|| / ||attn(q, K, V)||, queries q [M][L][d],
    K/V [N][L][d]."""
    out = []
    for l in range(K.shape[1]):
        o = O.softmax_attention(q[:, l], K[:, l], V[:, l], scale)
        oh = O.softmax_attention(q[:, l], Kh[:, l], Vh[:, l], scale)
        out.append(np.linalg.norm(oh - o) / np.linalg.norm(o))
    return np.array(out)
