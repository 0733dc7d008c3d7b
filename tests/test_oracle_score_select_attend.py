"""Pins of the oracle's score, selection and attention.

Score (CSA-indexer commit): sum_h relu(e4m3(q_h) . summary) * w_h over a KV group's
indexer heads, a contiguous block of them (provider groups).  Pinned by exact rational
arithmetic, hand-derived golden cases and special cases.
Selection: the K smallest (-score, id) keys, in key order; pinned by Python's sort and golden
cases.  Attention over the picks plus the row's own region; with every region picked
it is dense causal attention (torch's scaled_dot_product_attention in fp64 is the
independent library pin).
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def bf16_codes(vals):
    return torch.tensor(np.asarray(vals, dtype=np.float64), dtype=torch.float32).to(torch.bfloat16) \
        .view(torch.int16).numpy().view(np.uint16)


def e4m3_codes(vals):
    return torch.tensor(np.asarray(vals, dtype=np.float64), dtype=torch.float32) \
        .to(torch.float8_e4m3fn).view(torch.uint8).numpy()


# ---------------------------------------------------------------- score

def test_score_golden(orc):
    spec = json.load(open(os.path.join(GOLD, "score_cases.json")))
    q = np.zeros((4, 64), np.uint16)
    for h, dims in spec["q"].items():
        for d, v in dims.items():
            q[int(h), int(d)] = bf16_codes([v])[0]
    summ = np.zeros((len(spec["regions"]), 64), np.uint8)
    for r, reg in enumerate(spec["regions"]):
        for d, c in reg["summary"].items():
            summ[r, int(d)] = c
    got = orc.score_group(q, np.array(spec["w"], np.float32), 0, 32, summ)
    want = [reg["score"] for reg in spec["regions"]]
    assert list(got) == want
    assert not np.signbit(got[1])   # relu zero is +0


def test_score_exact_rational_bruteforce(orc):
    rng = np.random.default_rng(11)
    hpg, R = 4, 40
    q = bf16_codes(rng.standard_normal((hpg, 64)) * 4)
    w = rng.uniform(0, 1, hpg).astype(np.float32)
    summ = e4m3_codes(rng.standard_normal((R, 64)))
    pos = 77
    theta = (np.arange(128)[:, None] * 10000.0 ** (-np.arange(16) / 16.0))
    cos, sin = bf16_codes(np.cos(theta)), bf16_codes(np.sin(theta))
    got = orc.score_group(q, w, pos, 32, summ, cos, sin)
    # exact: rotated q (oracle rotation, pinned separately) -> e4m3 via torch's cast
    qe = []
    for h in range(hpg):
        rq = orc.rotate_neox(q[h], 32, cos[pos], sin[pos])
        qe.append([Fraction(float(v)) for v in torch.from_numpy(rq).to(torch.float32)
                   .to(torch.float8_e4m3fn).to(torch.float64).numpy()])
    sv = [[Fraction(orc.e4m3_value(int(c))) for c in row] for row in summ]
    for r in range(R):
        tot = Fraction(0)
        for h in range(hpg):
            dot = sum(qe[h][d] * sv[r][d] for d in range(64))
            tot += max(dot, Fraction(0)) * Fraction(float(w[h]))
        assert abs(got[r] - float(tot)) <= 1e-15 * abs(float(tot)) + 1e-300


def test_score_special_cases(orc):
    rng = np.random.default_rng(12)
    q = bf16_codes(rng.standard_normal((4, 64)))
    summ = e4m3_codes(rng.standard_normal((30, 64)))
    assert np.all(orc.score_group(q, np.zeros(4, np.float32), 5, 32, summ) == 0)
    assert np.all(orc.score_group(np.zeros((4, 64), np.uint16), np.ones(4, np.float32), 5, 32, summ) == 0)
    # flipping the summary's sign keeps only the heads that were clipped before
    w = np.ones(4, np.float32)
    a = orc.score_group(q, w, 5, 32, summ)
    b = orc.score_group(q, w, 5, 32, summ ^ np.uint8(0x80))
    qe = orc.e4m3_values(orc.bf16_codes_to_e4m3_codes(q))
    sv = orc.e4m3_values(summ)
    dots = sv @ qe.T
    assert np.allclose(a + b, np.abs(dots).sum(axis=1), rtol=1e-14)
    # linear in w
    w2 = rng.uniform(0, 1, 4).astype(np.float32)
    assert np.allclose(orc.score_group(q, 2 * w2, 5, 32, summ), 2 * orc.score_group(q, w2, 5, 32, summ), rtol=1e-15)


def test_score_batch_group_head_blocks(orc):
    # only heads 4..7 (group 1's contiguous block) non-zero -> only group 1 scores
    rng = np.random.default_rng(13)
    N, G, r_cap = 2, 4, 6
    q = np.zeros((N, 16, 64), np.uint16)
    q[:, 4:8] = bf16_codes(np.abs(rng.standard_normal((N, 4, 64))))
    w = np.ones((N, 16), np.float32)
    summ = e4m3_codes(np.abs(rng.standard_normal((1, G, r_cap, 64))))
    pos = np.array([40, 23], np.int32)
    seq = np.zeros(N, np.int32)
    scores, _ = orc.score_batch(q, w, seq, pos, summ, G, 32, nthreads=2)
    for n in range(N):
        R = pos[n] // 8
        for g in range(G):
            if g == 1:
                assert np.all(scores[n, g, :R] > 0)
                ref = orc.score_group(q[n, 4:8], w[n, 4:8], pos[n], 32, summ[0, 1, :R])
                assert np.array_equal(scores[n, g, :R], ref)
            else:
                assert np.all(scores[n, g, :R] == 0)
            assert np.all(np.isnan(scores[n, g, R:]))


# ---------------------------------------------------------------- select

def test_select_golden(orc):
    spec = json.load(open(os.path.join(GOLD, "select_cases.json")))
    for case in spec["cases"]:
        got = orc.select_topk(np.array(case["scores"], np.float64), case["K"])
        assert list(got) == case["ids"], case


@pytest.mark.parametrize("R,K", [(1, 512), (100, 512), (600, 512), (5000, 512), (64, 7)])
def test_select_vs_python_sort(orc, R, K):
    rng = np.random.default_rng(R + K)
    s = np.round(rng.standard_normal(R) * 4) / 4          # many exact ties
    s[rng.integers(0, R, R // 10 + 1)] = 0.0
    got = orc.select_topk(s, K)
    want = sorted(range(R), key=lambda i: (-s[i], i))[:K]
    assert list(got) == want


def test_select_all_equal_gives_first_ids(orc):
    assert list(orc.select_topk(np.zeros(2000), 512)) == list(range(512))


# ---------------------------------------------------------------- attend

def test_attend_golden(orc):
    spec = json.load(open(os.path.join(GOLD, "attend_cases.json")))
    for case in spec["cases"]:
        t_cap = 8 * (case["pos"] // 8 + 1)
        kc = np.zeros((t_cap, 128), np.uint16)
        vc = np.zeros((t_cap, 128), np.uint16)
        for t, v in case["k0"].items():
            kc[int(t), 0] = bf16_codes([v])[0]
        for t, v in case["v0"].items():
            vc[int(t), 0] = bf16_codes([v])[0]
        q = np.zeros((1, 128), np.uint16)
        q[0, 0] = bf16_codes([case["q0"]])[0]
        out = orc.attend_group(q, kc, vc, np.array(case["sel"], np.int32), case["pos"], 8, 1.0)
        want = eval(case["out0_formula"], {"exp": math.exp})
        assert abs(out[0, 0] - want) <= 1e-14 * abs(want), case["name"]
        assert np.all(out[0, 1:] == 0)


def test_attend_dense_equivalence_vs_sdpa(orc):
    """With every completed region picked, the output equals dense causal attention
    over tokens 0..pos (torch SDPA, fp64)."""
    rng = np.random.default_rng(21)
    hq, D = 8, 128
    for pos in (0, 7, 8, 9, 63, 100):
        t_cap = 8 * (pos // 8 + 1)
        q = bf16_codes(rng.standard_normal((hq, D)))
        kc = bf16_codes(rng.standard_normal((t_cap, D)))
        vc = bf16_codes(rng.standard_normal((t_cap, D)))
        sel = np.arange(pos // 8, dtype=np.int32)[::-1].copy()   # order must not matter
        out = orc.attend_group(q, kc, vc, sel, pos, 8, 1 / math.sqrt(D))
        qt = torch.from_numpy(orc.bf16_values(q))[None]
        kt = torch.from_numpy(orc.bf16_values(kc[:pos + 1]))[None, None].expand(1, hq, pos + 1, D)
        vt = torch.from_numpy(orc.bf16_values(vc[:pos + 1]))[None, None].expand(1, hq, pos + 1, D)
        ref = torch.nn.functional.scaled_dot_product_attention(qt[:, :, None, :].transpose(0, 1).reshape(1, hq, 1, D), kt, vt)
        assert np.allclose(out, ref[0, :, 0].numpy(), rtol=1e-12, atol=1e-12)


def test_attend_ignores_tokens_past_pos_and_unpicked(orc):
    rng = np.random.default_rng(22)
    hq, D, pos = 4, 128, 42
    t_cap = 48
    q = bf16_codes(rng.standard_normal((hq, D)))
    kc = bf16_codes(rng.standard_normal((t_cap, D)))
    vc = bf16_codes(rng.standard_normal((t_cap, D)))
    sel = np.array([3, 0], np.int32)
    out = orc.attend_group(q, kc, vc, sel, pos, 8, 0.1)
    kc2, vc2 = kc.copy(), vc.copy()
    nan = bf16_codes([np.nan])[0]
    kc2[pos + 1:] = nan
    vc2[pos + 1:] = nan
    kc2[8:24] = nan        # regions 1, 2: not picked
    vc2[8:24] = nan
    out2 = orc.attend_group(q, kc2, vc2, sel, pos, 8, 0.1)
    assert np.array_equal(out, out2)
