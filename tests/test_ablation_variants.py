"""Ablation rows on the CPU: each simplification of the method costs reconstruction error.

Seeded synthetic states with the layer_1p4b generator (outlier channel x10, inter-loop noise
0.1) and with gqa_deep's heavy-tailed one; each step the method adds must lower the error of
the non-final loops against the variant that drops it (averaged over a sample of tokens and
heads, K and V)."""

import dataclasses

import numpy as np
import pytest

import synth
from ablation import VARIANTS, bytes_per_token_head, rel_err

pytestmark = pytest.mark.filterwarnings("ignore")


def _errors(name, res_bits=None, n_tok=384, heads=(0, 1)):
    cfg = synth.config_by_name(name)
    if res_bits is not None:
        cfg = dataclasses.replace(cfg, res_bits=tuple(res_bits))
    rb = list(cfg.res_bits[: cfg.n_loops - 1])
    x = synth.gen_states(cfg, 0, [0], np.arange(n_tok), heads=list(heads))[0]   # [t][kv][L][h][d]
    signs = synth.rotation_signs(cfg, 0)
    err = {v: np.zeros(cfg.n_loops) for v in VARIANTS}
    for hi, h in enumerate(heads):
        for kv in range(2):
            xs = x[:, kv, :, hi, :].astype(np.float64)
            for v, f in VARIANTS.items():
                err[v] += rel_err(xs, f(xs, signs[h, kv].astype(np.float64), rb))
    n = 2 * len(heads)
    return {v: e / n for v, e in err.items()}, cfg


@pytest.mark.parametrize("name", ["layer_1p4b", "gqa_deep"])
def test_reference_and_ls_scale_lower_the_error(name):
    err, cfg = _errors(name)
    nf = slice(0, cfg.n_loops - 1)
    rq = err["rq"][nf]
    assert np.all(5 * rq < err["direct"][nf]), err      # the reference + residual beats direct INT2
    assert np.all(rq < err["no_ls"][nf]), err           # the LS scale
    assert np.allclose(err["rq"][-1], err["direct"][-1])   # same INT4 reference


def test_rotation_lowers_the_error_of_residuals_with_outlier_channels():
    # the synthetic generator's outliers sit in the base state, which the reference absorbs;
    # here the loop-to-loop difference itself has two outlier channels (x40), the case the
    # rotation is for: without it, the two groups holding them quantise their other 62
    # channels on a 40x wider step
    rng = np.random.default_rng(0)
    n, d = 512, 128
    b = rng.standard_normal((n, d))
    delta = 0.05 * rng.standard_normal((n, d))
    delta[:, 3] *= 40
    delta[:, 70] *= 40
    x = np.stack([b + delta, b], axis=1)
    signs = np.where(rng.random(d) < 0.5, -1.0, 1.0)
    e_rot = rel_err(x, VARIANTS["rq"](x, signs, [2]))[0]
    e_id = rel_err(x, VARIANTS["no_rotation"](x, signs, [2]))[0]
    assert e_rot < 0.85 * e_id, (e_rot, e_id)


def test_four_bit_residual_lowers_its_loop_error():
    all2, _ = _errors("layer_1p4b", res_bits=(2, 2, 2))
    mixed, _ = _errors("layer_1p4b", res_bits=(4, 2, 2))
    assert mixed["rq"][0] < 0.5 * all2["rq"][0]
    assert np.allclose(mixed["rq"][1:], all2["rq"][1:])


def test_bytes_of_the_variants():
    assert bytes_per_token_head("rq", 128, [2, 2, 2]) == 460
    assert bytes_per_token_head("direct", 128, [2, 2, 2]) == 448
    assert bytes_per_token_head("rq", 128, [4, 2, 2]) == 524
