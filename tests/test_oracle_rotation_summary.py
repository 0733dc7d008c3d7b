"""Pins of the oracle's NEOX rotation and region summary.

Rotation (the page's glue commit: q and k take NEOX rotation from bf16 cos/sin tables;
the indexer commit: on their first 32 dims): pairs (i, i + 16), x1' = x1 c - x2 s, x2' = x2 c + x1 s, rounded once to bf16.
Summary (CSA-indexer commit): s[d] = sum_t softmax_t(z[., d]) rot(k)[t][d], then
e4m3(bf16(s)).  Pinned by hand-derived golden cases, closed forms and the fp64
torch.softmax / einsum library path.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def bf16_codes(vals):
    return torch.tensor(vals, dtype=torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_rotation_identity_and_quarter_turn(orc):
    rng = np.random.default_rng(1)
    x = bf16_codes(rng.standard_normal(64))
    xv = orc.bf16_values(x)
    half = 16
    ones = bf16_codes(np.ones(half))
    zeros = bf16_codes(np.zeros(half))
    out = orc.rotate_neox(x, 32, ones, zeros)
    assert np.array_equal(out, xv)
    out = orc.rotate_neox(x, 32, zeros, ones)              # c = 0, s = 1
    assert np.array_equal(out[:16], -xv[16:32])            # x1' = -x2
    assert np.array_equal(out[16:32], xv[:16])             # x2' = x1
    assert np.array_equal(out[32:], xv[32:])               # dims >= 32 untouched
    assert np.array_equal(orc.rotate_neox(x, 32, None, None), xv)


def test_rotation_preserves_norm_and_inverts(orc):
    rng = np.random.default_rng(2)
    x = bf16_codes(rng.standard_normal(64))
    xv = orc.bf16_values(x)
    theta = rng.uniform(-3, 3, 16)
    c, s = bf16_codes(np.cos(theta)), bf16_codes(np.sin(theta))
    cv, sv = orc.bf16_values(c), orc.bf16_values(s)
    out = orc.rotate_neox(x, 32, c, s)
    # each pair's norm scales by (c^2 + s^2) (bf16 tables) up to two bf16 roundings
    for i in range(16):
        n0 = xv[i] ** 2 + xv[i + 16] ** 2
        n1 = out[i] ** 2 + out[i + 16] ** 2
        assert abs(n1 - n0 * (cv[i] ** 2 + sv[i] ** 2)) <= 4 * 2.0 ** -8 * (n0 + 1e-30)
    # rotating back by -theta recovers x to bf16 accuracy
    back = orc.rotate_neox(bf16_codes(out), 32, c, bf16_codes(-orc.bf16_values(s)))
    scale = np.concatenate([cv ** 2 + sv ** 2, cv ** 2 + sv ** 2, np.ones(32)])
    assert np.allclose(back, xv * scale, rtol=2e-2, atol=2e-2)


def test_rotation_single_rounding(orc):
    # x1 = 1 + 2^-7, c = 1 + 2^-7, x2 = 2^-7, s = 2^-8 (all bf16):
    # x1*c - x2*s = 1 + 2^-6 + 2^-14 - 2^-15 = 1 + 2^-6 + 2^-15 -> bf16 1 + 2^-6
    x = np.zeros(64, np.uint16)
    x[0] = bf16_codes([1 + 2 ** -7])[0]
    x[16] = bf16_codes([2 ** -7])[0]
    c = bf16_codes([1 + 2 ** -7] + [1.0] * 15)
    s = bf16_codes([2 ** -8] + [0.0] * 15)
    out = orc.rotate_neox(x, 32, c, s)
    assert out[0] == 1 + 2 ** -6
    # x2' = x2 c + x1 s = 2^-7 + 2^-14 + 2^-8 + 2^-15 -> bf16 (spacing 2^-14 at 2^-7)
    exact = 2 ** -7 * (1 + 2 ** -7) + (1 + 2 ** -7) * 2 ** -8
    assert out[16] == float(torch.tensor(exact, dtype=torch.float64).to(torch.bfloat16).double())


def _region(dim_vals_k, dim_vals_z, dim):
    k = np.zeros((8, 64), np.uint16)
    z = np.zeros((8, 64), np.uint16)
    k[:, dim] = bf16_codes(dim_vals_k)
    z[:, dim] = bf16_codes(dim_vals_z)
    return k, z


def test_summary_golden_cases(orc):
    spec = json.load(open(os.path.join(GOLD, "summary_cases.json")))
    for case in spec["cases"]:
        d = case["dim"]
        k, z = _region(case["k"], case["z"], d)
        s, code = orc.summarize_region(k, z, 0, 32, None, None)
        want = case["s"] if "s" in case else eval(case["s_formula"], {"exp": math.exp})
        tol = case.get("s_tol", 0.0)
        assert abs(s[d] - want) <= tol, case["name"]
        assert code[d] == case["code"], case["name"]
        others = [i for i in range(64) if i != d]
        assert np.all(s[others] == 0.0) and np.all(code[others] == 0), case["name"]
    for case in spec["rotated_cases"]:
        k = np.zeros((8, 64), np.uint16)
        z = np.zeros((8, 64), np.uint16)
        k[:, 0] = bf16_codes([case["k_dim0"]] * 8)
        k[:, 16] = bf16_codes([case["k_dim16"]] * 8)
        cos = np.tile(bf16_codes([case["cos"]] * 16), (8, 1))
        sin = np.tile(bf16_codes([case["sin"]] * 16), (8, 1))
        s, code = orc.summarize_region(k, z, 0, 32, cos, sin)
        assert s[0] == case["s_dim0"] and s[16] == case["s_dim16"], case["name"]
        assert code[0] == case["code_dim0"] and code[16] == case["code_dim16"], case["name"]


def test_summary_constant_z_is_mean_and_shift_invariant(orc):
    rng = np.random.default_rng(3)
    k = bf16_codes(rng.standard_normal((8, 64)))
    kv = orc.bf16_values(k)
    for zval in (0.0, 7.0, -30.0):
        z = bf16_codes(np.full((8, 64), zval))
        s, _ = orc.summarize_region(k, z, 0, 32, None, None)
        assert np.allclose(s, kv.mean(axis=0), rtol=0, atol=1e-15)


def test_summary_dominant_token(orc):
    rng = np.random.default_rng(4)
    k = bf16_codes(rng.standard_normal((8, 64)))
    kv = orc.bf16_values(k)
    zz = np.zeros((8, 64))
    winner = rng.integers(0, 8, 64)
    zz[winner, np.arange(64)] = 60.0
    s, _ = orc.summarize_region(k, bf16_codes(zz), 0, 32, None, None)
    assert np.allclose(s, kv[winner, np.arange(64)], rtol=0, atol=1e-20)


def test_summary_vs_torch_softmax_library(orc):
    rng = np.random.default_rng(6)
    t0 = 40
    k = bf16_codes(rng.standard_normal((8, 64)))
    z = bf16_codes(rng.standard_normal((8, 64)) * 2)
    theta = (np.arange(64)[:, None] * 10000.0 ** (-np.arange(16) / 16.0))
    cos, sin = bf16_codes(np.cos(theta)), bf16_codes(np.sin(theta))
    s, code = orc.summarize_region(k, z, t0, 32, cos, sin)
    # library path: rotate with the (pinned) oracle rotation, then torch fp64 softmax
    kr = np.stack([orc.rotate_neox(k[t], 32, cos[t0 + t], sin[t0 + t]) for t in range(8)])
    zt = torch.from_numpy(orc.bf16_values(z))
    w = torch.softmax(zt, dim=0)
    ref = torch.einsum("td,td->d", w, torch.from_numpy(kr)).numpy()
    assert np.allclose(s, ref, rtol=1e-13, atol=1e-15)
    ref_code = torch.from_numpy(ref).to(torch.float32).to(torch.bfloat16).to(torch.float8_e4m3fn)
    # fp64 -> fp32 -> bf16 can double-round; only compare where fp32 was exact enough
    okmask = np.abs(ref - ref.astype(np.float32)) < 1e-12 * np.abs(ref) + 1e-300
    assert np.array_equal(code[okmask], ref_code.view(torch.uint8).numpy()[okmask])


def test_summary_batch_matches_single(orc):
    rng = np.random.default_rng(7)
    B, G, t_cap, r_cap = 2, 4, 40, 5
    k = bf16_codes(rng.standard_normal((B, G, t_cap, 64)))
    z = bf16_codes(rng.standard_normal((B, G, t_cap, 64)))
    theta = (np.arange(t_cap)[:, None] * 10000.0 ** (-np.arange(16) / 16.0))
    cos, sin = bf16_codes(np.cos(theta)), bf16_codes(np.sin(theta))
    rb = np.array([1, 0], np.int32)
    re = np.array([4, 5], np.int32)
    summ, s64, _ = orc.summarize_batch(k, z, cos, sin, rb, re, r_cap, 32, want_f64=True, nthreads=3)
    for b in range(B):
        for g in range(G):
            for r in range(r_cap):
                if rb[b] <= r < re[b]:
                    s, c = orc.summarize_region(k[b, g, 8 * r:8 * r + 8], z[b, g, 8 * r:8 * r + 8],
                                                8 * r, 32, cos, sin)
                    assert np.array_equal(summ[b, g, r], c) and np.array_equal(s64[b, g, r], s)
                else:
                    assert np.all(summ[b, g, r] == 0)
