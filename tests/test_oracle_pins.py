"""Pins of the fp64 oracle against facts the method and the mathematics fix.

None of these re-types the oracle's formula: each compares it with a brute-force
search, a construction whose answer is known exactly, an invariant, a library routine
or a hand-derived closed form.
"""

import numpy as np
import pytest

import oracle as O

RNG = np.random.default_rng(1234)


def _states(N, L, d, sigma=0.1, rng=RNG):
    base = rng.standard_normal((N, 1, d))
    u = rng.uniform(0.8, 1.2, (N, L, 1))
    x = u * base + sigma * rng.standard_normal((N, L, d))
    return O.bf16_round(x)


def _signs(d, rng=RNG):
    return rng.choice([-1.0, 1.0], size=d)


# --------------------------------------------------------------------- rounding helpers

def _all_fp16_finite():
    v = np.arange(0, 0x7C00, dtype=np.uint16).view(np.float16).astype(np.float64)
    return np.concatenate([-v[::-1], v])


def test_fp16_round_is_nearest_ties_even():
    grid = np.unique(_all_fp16_finite())
    x = np.concatenate([RNG.standard_normal(2000) * 10, RNG.standard_normal(500) * 1e-5,
                        (grid[:-1] + grid[1:])[::97] / 2])   # exact midpoints included
    got = O.fp16_round(x)
    i = np.searchsorted(grid, x)
    lo, hi = grid[np.clip(i - 1, 0, len(grid) - 1)], grid[np.clip(i, 0, len(grid) - 1)]
    dlo, dhi = np.abs(x - lo), np.abs(hi - x)
    even_hi = (np.abs(hi.astype(np.float16).view(np.uint16).astype(int)) & 1) == 0
    want = np.where(dlo < dhi, lo, np.where(dhi < dlo, hi, np.where(even_hi, hi, lo)))
    assert np.array_equal(got, want)


def test_bf16_round_matches_torch_on_fp32_inputs():
    torch = pytest.importorskip("torch")
    x = np.concatenate([RNG.standard_normal(5000).astype(np.float32) * 3,
                        np.array([1.00390625, 1.01171875, -2.0078125], np.float32)])
    want = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(O.bf16_round(x.astype(np.float64)), want)


# --------------------------------------------------------------------- LS scale (step 3)

def _golden_min(f, a, b, iters=200):
    g = (np.sqrt(5) - 1) / 2
    c, d = b - g * (b - a), a + g * (b - a)
    for _ in range(iters):
        if f(c) < f(d):
            b = d
        else:
            a = c
        c, d = b - g * (b - a), a + g * (b - a)
    return (a + b) / 2


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_ls_scale_minimises_residual_norm_by_brute_force(seed):
    rng = np.random.default_rng(seed)
    x = _states(1, 4, 128, rng=rng)[0]
    enc = O.encode(x[None], _signs(128, rng), (2, 2, 2))
    ref_hat = O.dequant(*[e[0] for e in enc["ref"]])
    for l in range(3):
        xl = x[l]
        grid = np.arange(-400000, 400001) * 1e-5                     # [-4, 4] step 1e-5
        # ||x - a r||^2 expanded per grid point, in chunks to bound memory
        best, best_a = np.inf, None
        for c0 in range(0, grid.size, 100000):
            g = grid[c0:c0 + 100000]
            e = (xl @ xl) - 2 * g * (xl @ ref_hat) + g * g * (ref_hat @ ref_hat)
            k = int(np.argmin(e))
            if e[k] < best:
                best, best_a = e[k], g[k]
        f = lambda a: float(np.sum((xl - a * ref_hat) ** 2))
        a_star = _golden_min(f, best_a - 2e-5, best_a + 2e-5)
        a_cf = O.ls_scale(xl, ref_hat)
        # comparing values of a quadratic resolves its minimiser only to about sqrt(eps)
        assert abs(a_star - a_cf) < 1e-7
        a_h = enc["alpha"][l][0]
        f16 = np.sort(np.unique(_all_fp16_finite()))
        i = np.searchsorted(f16, a_star)
        assert a_h in (f16[i - 1], f16[i])


def test_ls_scale_zero_reference_gives_zero():
    assert O.ls_scale(np.ones(32), np.zeros(32)) == 0.0


# ---------------------------------------------------------------- residual (steps 3-4)

def _on_grid_reference(N, d, rng):
    """x on the INT4 grid: every group holds codes 0 and 15, s a power of two, z = k s."""
    ng = d // 32
    codes = rng.integers(0, 16, size=(N, ng, 32))
    codes[:, :, 0] = 0
    codes[:, :, 1] = 15
    for t in range(N):
        for g in range(ng):
            rng.shuffle(codes[t, g])
    s = 2.0 ** rng.integers(-6, 0, size=(N, ng, 1))
    z = rng.integers(-12, 3, size=(N, ng, 1)) * s
    return (codes * s + z).reshape(N, d)


def test_zero_noise_on_grid_gives_exactly_zero_residual():
    rng = np.random.default_rng(7)
    N, L, d = 16, 4, 128
    ref = _on_grid_reference(N, d, rng)
    assert np.array_equal(O.bf16_round(ref), ref)
    x = np.repeat(ref[:, None, :], L, axis=1)
    enc = O.encode(x, _signs(d, rng), (2, 4, 2))
    assert np.array_equal(O.dequant(*enc["ref"]), ref)          # reference is lossless
    for l in range(L - 1):
        assert np.all(enc["alpha"][l] == 1.0)
        c, s, z = enc["res"][l]
        assert np.all(c == 0) and np.all(s == 0) and np.all(z == 0)
    assert np.array_equal(O.reconstruct(enc, _signs(d, rng)), x)


def test_reference_is_the_final_loop():
    rng = np.random.default_rng(3)
    x = _states(8, 4, 64, rng=rng)
    enc = O.encode(x, _signs(64, rng), (2, 2, 2))
    for l in range(3):
        c_l, _, _ = O.quantize(x[:, l, :], 4, "t")
        assert not np.array_equal(c_l, enc["ref"][0])
    c_f, s_f, z_f = O.quantize(x[:, 3, :], 4, "t")
    assert np.array_equal(c_f, enc["ref"][0])
    assert np.array_equal(O.reconstruct(enc, _signs(64, rng))[:, 3, :], O.dequant(c_f, s_f, z_f))


# -------------------------------------------------------------- INT2 / INT4 (steps 2, 6)

@pytest.mark.parametrize("bits", [2, 4])
def test_min_max_quantiser_uses_all_levels_and_bounds_error(bits):
    v = RNG.standard_normal((4000, 64)) * RNG.uniform(0.1, 10, (4000, 1))
    c, s_h, z_h = O.quantize(v, bits, "t")
    g = O.group_view(v)
    cg = O.group_view(c)
    am, ax = g.argmin(-1), g.argmax(-1)
    assert np.all(np.take_along_axis(cg, am[..., None], -1) == 0)
    assert np.all(np.take_along_axis(cg, ax[..., None], -1) == 2 ** bits - 1)
    assert set(np.unique(c).astype(int)) == set(range(2 ** bits))
    deq = O.group_view(O.dequant(c, s_h, z_h))
    top = (z_h + (2 ** bits - 1) * s_h)[..., None]
    unclamped = (g >= z_h[..., None]) & (g <= top)
    err = np.abs(g - deq)
    assert np.all(err[unclamped] <= (s_h[..., None] / 2 * (1 + 1e-12) + 0 * g)[unclamped])
    lo_bound = np.abs(g.min(-1) - z_h)[..., None] + 0 * g
    hi_bound = np.abs(g.max(-1)[..., None] - top) + 0 * g
    assert np.all(err[~unclamped] <= np.maximum(lo_bound, hi_bound)[~unclamped] + 1e-15)


def test_constant_group_dequantises_to_offset():
    v = np.full((1, 32), 0.3125)
    c, s_h, z_h = O.quantize(v, 2, "t")
    assert np.all(c == 0) and s_h[0, 0] == 0 and z_h[0, 0] == 0.3125
    assert np.all(O.dequant(c, s_h, z_h) == 0.3125)


# ------------------------------------------------------------------------- rotation (5)

def _fwht(v):
    v = np.array(v, dtype=np.float64)
    h = 1
    while h < v.shape[-1]:
        a = v.reshape(v.shape[:-1] + (-1, 2, h))
        x, y = a[..., 0, :].copy(), a[..., 1, :].copy()
        a[..., 0, :], a[..., 1, :] = x + y, x - y
        v = a.reshape(v.shape)
        h *= 2
    return v


@pytest.mark.parametrize("d", [64, 128])
def test_rotation_is_orthogonal_and_equals_fwht(d):
    s = _signs(d)
    R = O.rotation(s)
    assert np.max(np.abs(R @ R.T - np.eye(d))) < 1e-14
    v = RNG.standard_normal((5, d))
    assert np.max(np.abs(v @ R.T - _fwht(v * s) / np.sqrt(d))) < 1e-13


def test_rotation_applies_signs_before_hadamard():
    """R e_0 = s_0 H[:, 0] / sqrt(d) is constant (H's first column is all ones); the
    transposed order (H after... signs last) would give the sign vector instead."""
    s = _signs(64)
    s[0] = -1.0
    e0 = np.zeros(64)
    e0[0] = 1.0
    assert np.allclose(O.rotation(s) @ e0, -np.ones(64) / 8.0, atol=0, rtol=1e-15)


def test_attention_invariant_to_rotating_query_and_output():
    rng = np.random.default_rng(11)
    N, L, d = 300, 4, 128
    xk, xv = _states(N + 1, L, d, rng=rng), _states(N + 1, L, d, rng=rng)
    sk, sv = _signs(d, rng), _signs(d, rng)
    ek = O.encode(xk[:N], sk, (4, 2, 2))
    ev = O.encode(xv[:N], sv, (4, 2, 2))
    q = O.bf16_round(rng.standard_normal((3, d)))
    for loop in range(L):
        a = O.decode_explicit(q, ek, ev, sk, sv, loop, xk[N, loop], xv[N, loop])
        b = O.decode_rotated(q, ek, ev, sk, sv, loop, xk[N, loop], xv[N, loop])
        assert np.max(np.abs(a - b)) < 1e-12


# ------------------------------------------------------------------------ attention (9)

def test_two_token_attention_by_hand():
    """ctx = 1 plus one pending token: out = p0 v0 + p1 v1, p = softmax of two scores."""
    rng = np.random.default_rng(5)
    d = 64
    xk, xv = _states(1, 1, d, rng=rng), _states(1, 1, d, rng=rng)     # L = 1: INT4 only
    ek = O.encode(xk, _signs(d), ())
    ev = O.encode(xv, _signs(d), ())
    k0 = O.dequant(*ek["ref"])[0]
    v0 = O.dequant(*ev["ref"])[0]
    k1, v1 = O.bf16_round(rng.standard_normal(d)), O.bf16_round(rng.standard_normal(d))
    q = O.bf16_round(rng.standard_normal(d))
    s0 = sum(q[i] * k0[i] for i in range(d)) / 8.0
    s1 = sum(q[i] * k1[i] for i in range(d)) / 8.0
    p0 = 1.0 / (1.0 + np.exp(s1 - s0))
    want = [p0 * v0[i] + (1.0 - p0) * v1[i] for i in range(d)]
    for f in (O.decode_explicit, O.decode_rotated):
        got = f(q[None], ek, ev, _signs(d), _signs(d), 0, k1, v1)
        assert np.max(np.abs(got[0] - np.array(want))) < 1e-13


def _lossless(name, pre, rounded):
    return pre if name.startswith(("res", "alpha")) else rounded


def test_lossless_residual_reconstructs_states_and_matches_sdpa():
    """With residuals kept in fp64 (no rounding anywhere after the reference), every loop
    is rebuilt exactly for any R, and attention equals library SDPA on the raw states."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(9)
    N, L, d = 200, 4, 128
    xk, xv = _states(N, L, d, rng=rng), _states(N, L, d, rng=rng)
    sk, sv = _signs(d, rng), _signs(d, rng)
    ek = O.encode(xk, sk, (2, 2, 2), rnd=_lossless)
    ev = O.encode(xv, sv, (2, 2, 2), rnd=_lossless)
    rk, rv = O.reconstruct(ek, sk), O.reconstruct(ev, sv)
    assert np.max(np.abs(rk[:, :3] - xk[:, :3])) < 1e-12
    assert np.max(np.abs(rv[:, :3] - xv[:, :3])) < 1e-12
    q = rng.standard_normal((4, d))
    for loop in range(3):
        got = O.decode_rotated(q, ek, ev, sk, sv, loop)
        ref = torch.nn.functional.scaled_dot_product_attention(
            torch.from_numpy(q)[None, None], torch.from_numpy(xk[:, loop])[None, None],
            torch.from_numpy(xv[:, loop])[None, None])[0, 0].numpy()
        assert np.max(np.abs(got - ref)) < 1e-12


def test_single_loop_reduces_to_int4_attention():
    rng = np.random.default_rng(2)
    N, d = 50, 64
    xk, xv = _states(N, 1, d, rng=rng), _states(N, 1, d, rng=rng)
    ek, ev = O.encode(xk, _signs(d), ()), O.encode(xv, _signs(d), ())
    q = rng.standard_normal((2, d))
    K = O.dequant(*O.quantize(xk[:, 0], 4, "t"))
    V = O.dequant(*O.quantize(xv[:, 0], 4, "t"))
    want = O.softmax_attention(q, K, V, 1 / 8.0)
    assert np.max(np.abs(O.decode_rotated(q, ek, ev, _signs(d), _signs(d), 0) - want)) < 1e-13


# ----------------------------------------------------------------------------- packing

@pytest.mark.parametrize("bits", [2, 4])
def test_pack_unpack_round_trip_and_bit_positions(bits):
    c = RNG.integers(0, 2 ** bits, size=(6, 128))
    rows = O.pack_rows(c, bits)
    assert rows.shape == (6, 128 * bits // 8)
    assert np.array_equal(O.unpack_rows(rows, bits, 128), c)
    one = np.zeros((1, 128), int)
    one[0, 5] = 1                              # channel 5 -> byte 5*b//8, bit (5*b)%8
    r = O.pack_rows(one, bits)
    assert r[0, 5 * bits // 8] == 1 << ((5 * bits) % 8) and r.sum() == r[0, 5 * bits // 8]
    rb = rows.shape[1]
    units = rb // 2
    phys = O.v_layout(rows)
    sw = int(O.v_unit_swizzle(1, units))                        # pair 1 = tokens 2, 3
    assert phys[1, 4 * sw:4 * sw + 2].tolist() == rows[2, 0:2].tolist()      # unit 0, token 2
    assert phys[1, 4 * sw + 2:4 * sw + 4].tolist() == rows[3, 0:2].tolist()  # unit 0, token 3
    u1 = 1 ^ sw
    assert phys[1, 4 * u1:4 * u1 + 2].tolist() == rows[2, 2:4].tolist()      # unit 1, token 2
    assert np.array_equal(O.v_unlayout(phys, rb), rows)
    # K rows: the k-th words of all groups are adjacent
    k = O.k_layout(rows, bits, 128)
    ng = 4
    assert k[0, 4:8].tolist() == rows[0, 4 * bits:4 * bits + 4].tolist()   # group 1, word 0
    assert np.array_equal(O.k_unlayout(k, bits, 128), rows)


@pytest.mark.parametrize("d,bits", [(64, (2, 2, 2)), (128, (4, 2, 2)), (128, (2,) * 7)])
def test_cache_bytes_matches_packed_arrays(d, bits):
    N = 10
    x = _states(N, len(bits) + 1, d)
    enc = O.encode(x, _signs(d), bits)
    n = O.pack_rows(enc["ref"][0], 4).size + 2 * enc["ref"][1].size * 2
    for l, (c, s, z) in enumerate(enc["res"]):
        n += O.pack_rows(c, bits[l]).size + 2 * s.size * 2 + 2 * enc["alpha"][l].size
    assert O.cache_bytes(d, len(bits) + 1, bits, N) == 2 * n
