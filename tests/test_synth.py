"""The shared seeded generator: Philox known answers and the state model's statistics."""

import os

import numpy as np

import synth
from synth.philox import philox4x32_10

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "philox_kat.txt")


def test_philox_known_answers():
    rows = [l.split() for l in open(GOLDEN) if l.strip() and not l.startswith("#")]
    assert len(rows) == 3
    for r in rows:
        v = [int(x, 16) for x in r]
        got = philox4x32_10(v[0], v[1], v[2], v[3], v[4], v[5])
        assert [int(g) for g in got] == v[6:]


def test_irwin_hall_normal_moments_and_determinism():
    c = synth.config_by_name("layer_1p4b")
    x = synth.gen_states(c, 0, [0, 1], np.arange(512), heads=[0, 5])
    y = synth.gen_states(c, 0, [0, 1], np.arange(512), heads=[0, 5])
    assert np.array_equal(x, y)
    # loops of one token are highly similar: u_l * base + small noise
    corr = np.corrcoef(x[:, :, 0, 0].ravel(), x[:, :, 0, 3].ravel())[0, 1]
    assert corr > 0.95
    q = synth.gen_queries(c, 0, np.arange(16))
    assert abs(q.mean()) < 0.01 and abs(q.std() - 1) < 0.01
    # every value is a bf16
    b = x.view(np.uint32)
    assert np.all((b & 0xFFFF) == 0)


def test_outliers_and_signs():
    c = synth.config_by_name("gqa_deep")
    ch = synth.outlier_channels(c, 0, 2, 1)
    assert len(ch) == 3 and len(set(ch)) == 3
    x = synth.gen_states(c, 0, [0], np.arange(2048), heads=[2], kvs=(1,))
    rms = np.sqrt((x[0, :, 0, 0, 0, :] ** 2).mean(axis=0))
    top = sorted(np.argsort(rms)[-3:].tolist())
    assert top == sorted(ch)
    s = synth.rotation_signs(c, 0)
    assert set(np.unique(s).tolist()) == {-1, 1} and abs(s.mean()) < 0.1


def test_subranges_are_consistent():
    c = synth.config_by_name("pr1_small")
    full = synth.gen_states(c, 0, [0], np.arange(64))
    part = synth.gen_states(c, 0, [0], np.arange(10, 20), heads=[1], loops=[2, 3], kvs=(1,))
    assert np.array_equal(part[0, :, 0, :, 0], full[0, 10:20, 1, 2:4, 1])
