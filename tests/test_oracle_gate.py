"""Pins of the oracle's per-head sigmoid output gate (the step after attention in the
Step-5 glue, which lists a per-head sigmoid gate).  Reading: one bf16 logit per (row, query
head); every output dim of the head is scaled by sigmoid(logit) before the output's one
bf16 rounding.  Pinned by closed forms: sigmoid(0) = 1/2 exactly, sigmoid(g) +
sigmoid(-g) = 1, sigmoid(1) = e / (1 + e), saturation at large |g|, and head
independence.
"""
import numpy as np

import oracle
import synthetic as S
import torch


def _out(seed, N=3, Hq=8, D=128):
    rng = np.random.default_rng(seed)
    return rng.standard_normal((N, Hq, D))


def _codes(values):
    return S.codes16(torch.tensor(values, dtype=torch.bfloat16))


def test_zero_logit_halves_exactly():
    o = _out(1)
    g = _codes(np.zeros((3, 8)))
    assert np.array_equal(oracle.sigmoid_gate(o, g), o * 0.5)


def test_opposite_logits_sum_to_the_ungated_output():
    o = _out(2)
    rng = np.random.default_rng(5)
    gv = rng.standard_normal((3, 8)) * 3
    gp = oracle.sigmoid_gate(o, _codes(gv))
    gn = oracle.sigmoid_gate(o, _codes(-gv))
    assert np.allclose(gp + gn, o, rtol=1e-14, atol=1e-15)
    # and the gate scales, never flips: same sign, smaller magnitude
    assert np.all(np.sign(gp) == np.sign(o)) and np.all(np.abs(gp) <= np.abs(o))


def test_logit_one_is_e_over_one_plus_e():
    o = _out(3)
    g = _codes(np.ones((3, 8)))
    assert np.allclose(oracle.sigmoid_gate(o, g), o * 0.7310585786300049, rtol=1e-15, atol=0)


def test_saturation():
    o = _out(4)
    assert np.array_equal(oracle.sigmoid_gate(o, _codes(np.full((3, 8), 88.0))), o)
    tiny = oracle.sigmoid_gate(o, _codes(np.full((3, 8), -88.0)))
    assert np.all(np.abs(tiny) <= np.abs(o) * 1e-37)


def test_each_head_uses_its_own_logit():
    o = _out(5)
    gv = np.full((3, 8), 88.0)
    gv[1, 5] = 0.0
    got = oracle.sigmoid_gate(o, _codes(gv))
    want = o.copy()
    want[1, 5] *= 0.5
    assert np.array_equal(got, want)
