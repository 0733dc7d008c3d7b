"""Pins of the oracle's indexer front end (CSA-indexer commit: the indexer's 16-head q
takes an RMSNorm with weight 1 + w, its k a LayerNorm with bias), by closed forms of the two norms
(constant, +-1 and 3-4 inputs, power-of-two scale and shift invariance) and by the
front end's composition: its caches and summaries are those of the separate steps, and
a region is summarised exactly when its last token arrives.
"""
import math

import numpy as np
import torch

import oracle
import synthetic as S


def codes(v):
    return S.codes16(torch.tensor(np.asarray(v, dtype=np.float32), dtype=torch.bfloat16))


def vals(c):
    return torch.from_numpy(np.asarray(c, dtype=np.uint16).view(np.int16).copy()).view(torch.bfloat16).float().numpy()


def test_rmsnorm_of_a_constant_is_one_plus_w():
    w = codes(np.linspace(-0.5, 0.5, 64))
    for c in (3.0, -0.25):
        y = vals(oracle.rmsnorm_1pw(codes(np.full(64, c)), w, eps=0.0))
        want = vals(codes(np.sign(c) * (1.0 + vals(w))))
        assert np.array_equal(y, want)


def test_rmsnorm_three_four():
    # mean of squares 12.5, so y = (3, 4) / (5 / sqrt 2) * (1 + w)
    x = codes([3.0, 4.0])
    w = codes([0.0, 1.0])
    y = vals(oracle.rmsnorm_1pw(x, w, eps=0.0))
    r2 = math.sqrt(2.0)
    assert np.array_equal(y, vals(codes([3 * r2 / 5, 2 * 4 * r2 / 5])))


def test_rmsnorm_is_scale_free():
    rng = np.random.default_rng(1)
    x = rng.standard_normal(64)
    w = codes(rng.standard_normal(64) * 0.1)
    a = oracle.rmsnorm_1pw(codes(x), w, eps=0.0)
    for s in (0.25, 8.0):
        assert np.array_equal(oracle.rmsnorm_1pw(codes(vals(codes(x)) * s), w, eps=0.0), a)


def test_layernorm_of_a_constant_is_the_bias():
    g = codes(np.linspace(0.5, 1.5, 64))
    b = codes(np.linspace(-1, 1, 64))
    y = oracle.layernorm(codes(np.full(64, 2.5)), g, b, eps=1e-6)
    assert np.array_equal(y, b)


def test_layernorm_plus_minus_one():
    x = codes(np.tile([1.0, -1.0], 32))  # mean 0, variance 1
    rng = np.random.default_rng(2)
    g = codes(rng.standard_normal(64))
    b = codes(rng.standard_normal(64))
    y = vals(oracle.layernorm(x, g, b, eps=0.0))
    want = vals(codes(vals(x) * vals(g) + vals(b)))
    assert np.array_equal(y, want)


def test_layernorm_is_shift_free():
    rng = np.random.default_rng(3)
    x = np.round(rng.standard_normal(64) * 8) / 8  # exact in bf16, and after +16
    g, b = codes(rng.standard_normal(64)), codes(rng.standard_normal(64))
    assert np.array_equal(oracle.layernorm(codes(x), g, b, 1e-6), oracle.layernorm(codes(x + 16.0), g, b, 1e-6))


def test_front_end_composes_the_steps_and_summarises_on_completion():
    rng = np.random.default_rng(4)
    G, H, D, B, t_cap, r_cap = 4, 16, 64, 2, 64, 8
    positions = np.array([15, 20], dtype=np.int32)  # row 0 completes region 1; row 1 does not
    seqs = np.array([0, 1], dtype=np.int32)
    q_pre = codes(rng.standard_normal((2, H, D)))
    k_pre = codes(rng.standard_normal((2, G, D)))
    z_pre = codes(rng.standard_normal((2, G, D)))
    qw, kw, kb = codes(rng.standard_normal(D) * 0.1), codes(1 + rng.standard_normal(D) * 0.1), codes(rng.standard_normal(D) * 0.1)
    kc = codes(rng.standard_normal((B, G, t_cap, D)))
    zc = codes(rng.standard_normal((B, G, t_cap, D)))
    ang = np.outer(np.arange(t_cap), 10000.0 ** (-np.arange(16) * 2 / 32))
    cos, sin = codes(np.cos(ang)), codes(np.sin(ang))
    summ = np.zeros((B, G, r_cap, D), dtype=np.uint8)
    q_out, kc2, zc2, summ2 = oracle.indexer_front(q_pre, k_pre, z_pre, qw, kw, kb, seqs, positions, cos, sin,
                                                  kc, zc, summ, eps=1e-6, rope_dims=32)
    assert np.array_equal(q_out, oracle.rmsnorm_1pw(q_pre, qw, 1e-6))
    for n in range(2):
        b, p = seqs[n], positions[n]
        assert np.array_equal(kc2[b, :, p], oracle.layernorm(k_pre[n], kw, kb, 1e-6))
        assert np.array_equal(zc2[b, :, p], z_pre[n])
        other = np.ones(t_cap, bool)
        other[p] = False
        assert np.array_equal(kc2[b][:, other], kc[b][:, other])
    # row 0 (p = 15) completed region 1: its summary is step (1) on the updated caches
    want, _, _ = oracle.summarize_batch(kc2, zc2, cos, sin, np.array([1, 0], np.int32), np.array([2, 0], np.int32),
                                        r_cap, 32, summ=summ.copy())
    assert np.array_equal(summ2, want)
    assert summ2[1].max() == 0  # row 1 (p = 20) completed nothing
