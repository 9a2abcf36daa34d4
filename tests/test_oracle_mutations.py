"""The oracle's pins catch plausible mistakes: each case plants one mistake in the oracle
(on the CPU, by replacing one of its functions) and checks that some pin fails."""

import numpy as np
import pytest

import oracle as O
import oracle.rq_oracle as R
import test_oracle_pins as pins

PIN_TESTS = [
    lambda: pins.test_fp16_round_is_nearest_ties_even(),
    lambda: pins.test_ls_scale_minimises_residual_norm_by_brute_force(0),
    lambda: pins.test_zero_noise_on_grid_gives_exactly_zero_residual(),
    lambda: pins.test_reference_is_the_final_loop(),
    lambda: pins.test_min_max_quantiser_uses_all_levels_and_bounds_error(2),
    lambda: pins.test_min_max_quantiser_uses_all_levels_and_bounds_error(4),
    lambda: pins.test_constant_group_dequantises_to_offset(),
    lambda: pins.test_rotation_is_orthogonal_and_equals_fwht(64),
    lambda: pins.test_rotation_applies_signs_before_hadamard(),
    lambda: pins.test_attention_invariant_to_rotating_query_and_output(),
    lambda: pins.test_two_token_attention_by_hand(),
    lambda: pins.test_lossless_residual_reconstructs_states_and_matches_sdpa(),
    lambda: pins.test_single_loop_reduces_to_int4_attention(),
    lambda: pins.test_pack_unpack_round_trip_and_bit_positions(2),
]


def _orig(name):
    return getattr(R, name)


def _mut_dequant_drops_offset():
    def f(c, s_h, z_h):
        g = R.group_view(c)
        return (g * s_h[..., None]).reshape(np.shape(c))
    return "dequant", f


def _mut_levels_2b():
    def f(v, bits):
        g = R.group_view(v)
        return (g.max(-1) - g.min(-1)) / (2 ** bits), g.min(-1)
    return "step_offset", f


def _mut_floor_codes():
    return "codes_from_quotient", lambda q, bits: np.clip(np.floor(q), 0, 2 ** bits - 1)


def _mut_rotation_transposed():
    o = _orig("rotation")
    return "rotation", lambda s: o(s).T


def _mut_ls_unscaled():
    return "ls_scale", lambda x, r: np.ones(np.shape(x)[:-1])


def _mut_ls_wrong_denominator():
    o = _orig("ls_scale")
    return "ls_scale", lambda x, r: o(x, r) * 1.01


def _mut_fp16_via_truncation():
    def f(x):
        x = np.asarray(x, np.float64)
        m, e = np.frexp(x)
        return np.ldexp(np.trunc(np.ldexp(m, 11)), e - 11)
    return "fp16_round", f


def _mut_decode_uses_transposed_rotation():
    o = _orig("decode_rotated")

    def f(*args, **kw):
        rot = R.rotation
        R.rotation = lambda sg: rot(sg).T      # R^T q instead of R q, R out instead of R^T
        try:
            return o(*args, **kw)
        finally:
            R.rotation = rot
    return "decode_rotated", f


def _mut_pack_big_endian():
    def f(codes, bits):
        c = np.asarray(codes).astype(np.uint32)
        N, d = c.shape
        per = 8 // bits
        c = c.reshape(N, d // per, per)
        out = np.zeros((N, d // per), dtype=np.uint32)
        for j in range(per):
            out |= c[:, :, j] << np.uint32(bits * (per - 1 - j))
        return out.astype(np.uint8)
    return "pack_rows", f


def _mut_softmax_scale():
    o = _orig("softmax_attention")
    return "softmax_attention", lambda q, K, V, scale: o(q, K, V, scale * 2)


MUTATIONS = [_mut_dequant_drops_offset, _mut_levels_2b, _mut_floor_codes,
             _mut_rotation_transposed, _mut_ls_unscaled, _mut_ls_wrong_denominator,
             _mut_fp16_via_truncation, _mut_decode_uses_transposed_rotation, _mut_pack_big_endian,
             _mut_softmax_scale]


@pytest.mark.parametrize("mutation", MUTATIONS, ids=lambda m: m.__name__[5:])
def test_planted_mistake_fails_a_pin(mutation, monkeypatch):
    name, fn = mutation()
    monkeypatch.setattr(R, name, fn)          # calls inside the oracle module
    monkeypatch.setattr(O, name, fn)          # calls through the package, as the pins make
    failed = []
    for t in PIN_TESTS:
        try:
            t()
        except (AssertionError, ValueError, FloatingPointError):
            failed.append(t)
    assert failed, "no pin caught the planted mistake in %s" % name
