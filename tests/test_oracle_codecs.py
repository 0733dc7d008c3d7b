"""Pins of the oracle's codecs against the format definitions and library casts.

bf16: nearest binary32 value with 7 stored mantissa bits, ties to even (the torch
fp32 -> bf16 cast is an independent implementation).  e4m3: OCP FP8 E4M3 "fn"
(bias 7, max 448, subnormal spacing 2^-9), saturating; pinned by brute-force
nearest search over the 254 finite codes and by torch's float8_e4m3fn cast.
"""
import numpy as np
import pytest
import torch


def _finite_e4m3_table(orc):
    codes = [c for c in range(256) if (c & 0x7F) != 0x7F]
    vals = np.array([orc.e4m3_value(c) for c in codes])
    return np.array(codes), vals


def test_e4m3_decode_matches_torch():
    import oracle
    torch_vals = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for c in range(256):
        v = oracle.e4m3_value(c)
        if (c & 0x7F) == 0x7F:
            assert np.isnan(v) and np.isnan(torch_vals[c])
        else:
            assert v == torch_vals[c], c
            assert np.signbit(v) == bool(c & 0x80)


def test_e4m3_decode_definition_spot_values(orc):
    assert orc.e4m3_value(0x7E) == 448.0
    assert orc.e4m3_value(0x08) == 2.0 ** -6          # min normal
    assert orc.e4m3_value(0x01) == 2.0 ** -9          # min subnormal
    assert orc.e4m3_value(0x07) == 7 * 2.0 ** -9      # max subnormal
    assert orc.e4m3_value(0x38) == 1.0
    assert orc.e4m3_value(0xC4) == -3.0


def test_e4m3_all_bf16_patterns_vs_bruteforce(orc):
    codes = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    x = orc.bf16_values(codes)
    finite = np.isfinite(x)
    got = orc.bf16_codes_to_e4m3_codes(codes)
    tcodes, tvals = _finite_e4m3_table(orc)
    # brute force: nearest finite e4m3 value; ties -> even mantissa; beyond 448 -> 448
    xf = x[finite]
    xs = np.clip(xf, -448.0, 448.0)
    dist = np.abs(xs[:, None] - tvals[None, :])
    best = dist.min(axis=1)
    expect = np.empty(xs.size, dtype=np.uint8)
    for i in range(xs.size):
        cand = np.nonzero(dist[i] == best[i])[0]
        cc = tcodes[cand]
        vv = tvals[cand]
        distinct = sorted(set(vv.tolist()))
        if len(distinct) == 2:
            # a tie between two values: the one whose mantissa field is even
            even_vals = [v for v, c in zip(vv, cc) if (c & 1) == 0]
            value = even_vals[0]
        else:
            value = distinct[0]
        if value == 0:
            # zero keeps the sign of x
            pick = 0x80 if np.signbit(xf[i]) else 0x00
        else:
            pick = [c for v, c in zip(vv, cc) if v == value][0]
        expect[i] = pick
    assert np.array_equal(got[finite], expect)
    # non-finite bf16 inputs: inf saturates, NaN stays NaN
    for c in codes[~finite]:
        v = orc.bf16_value(int(c))
        e = orc.e4m3_code(orc.round_e4m3(v))
        if np.isnan(v):
            assert (e & 0x7F) == 0x7F
        else:
            assert orc.e4m3_value(e) == np.sign(v) * 448.0


def test_e4m3_vs_torch_cast_in_range(orc):
    codes = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    x = orc.bf16_values(codes)
    ok = np.isfinite(x) & (np.abs(x) <= 448.0)
    got = orc.bf16_codes_to_e4m3_codes(codes[ok])
    t = torch.from_numpy(codes[ok].view(np.int16)).view(torch.bfloat16)
    ref = t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(got, ref)


def test_bf16_rounding_vs_fp32_cast(orc):
    rng = np.random.default_rng(5)
    vals = np.concatenate([
        rng.standard_normal(20000).astype(np.float32),
        (rng.standard_normal(2000) * 1e-38).astype(np.float32),      # subnormal range
        (rng.standard_normal(2000) * 1e30).astype(np.float32),
    ])
    # exact ties: bf16 value + half a bf16 ulp
    base = torch.from_numpy(rng.standard_normal(3000).astype(np.float32)).to(torch.bfloat16)
    b32 = base.to(torch.float32).numpy()
    ulp = np.abs(b32) * 2.0 ** -7
    ties = (b32 + np.sign(b32) * 0.5 * 2.0 ** np.floor(np.log2(np.abs(b32) + 1e-45)) * 2.0 ** -7).astype(np.float32)
    vals = np.concatenate([vals, ties, np.float32([0.0, -0.0, 1.0, 3.4e38, -3.4e38])])
    ref = torch.from_numpy(vals).to(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([orc.round_bf16(float(v)) for v in vals])
    assert np.array_equal(got, ref)
    assert np.array_equal(np.signbit(got), np.signbit(ref))
    del ulp


def test_bf16_rounding_of_fp64_is_single_rounding(orc):
    # 1 + 2^-8 + 2^-40 lies just above the bf16 midpoint 1 + 2^-8: correct rounding
    # goes up; rounding through fp32 first would land on the midpoint and go to even (1.0)
    x = 1.0 + 2.0 ** -8 + 2.0 ** -40
    assert orc.round_bf16(x) == 1.0 + 2.0 ** -7
    assert orc.round_bf16(1.0 + 2.0 ** -8) == 1.0          # exact tie -> even
    assert orc.round_bf16(1.0 + 3 * 2.0 ** -8) == 1.0 + 2.0 ** -6  # tie -> even (up)


def test_e4m3_code_roundtrip(orc):
    for c in range(256):
        if (c & 0x7F) == 0x7F:
            continue
        assert orc.e4m3_code(orc.e4m3_value(c)) == c
