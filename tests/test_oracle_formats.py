"""Pins of the oracle's number formats against library casts and exact brute force.

The oracle decodes and encodes E2M1 / E8M0 / E4M3 / BF16 from their bit fields
(oracle/formats.py). These tests check it against independent implementations: torch's
float8_e4m3fn / float8_e8m0fnu / bfloat16 casts, ml_dtypes' float4_e2m1fn where that
package is installed, and exact enumeration of representable neighbours.
"""

import numpy as np
import pytest
import torch

from oracle import formats as F

# OCP MX table of E2M1 values, codes 0..15 (sign bit 3)
E2M1_TABLE = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0,
              -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0]


def test_e2m1_all_codes_table():
    got = F.e2m1_to_float(np.arange(16))
    assert np.array_equal(got, np.array(E2M1_TABLE))
    assert np.array_equal(np.signbit(got[8:]), np.ones(8, bool)) or np.all(got[9:] < 0)


def test_e2m1_all_codes_ml_dtypes():
    ml = pytest.importorskip("ml_dtypes")
    vals = np.array(E2M1_TABLE, dtype=np.float32)
    codes = vals.astype(ml.float4_e2m1fn).view(np.uint8) & 0xF
    # ml_dtypes maps -0.0 to code 8
    assert np.array_equal(F.e2m1_to_float(codes), vals.astype(np.float64))
    back = np.arange(16, dtype=np.uint8).view(ml.float4_e2m1fn).astype(np.float32)
    assert np.array_equal(back.astype(np.float64), F.e2m1_to_float(np.arange(16)))


def test_e8m0_all_codes_torch():
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e8m0fnu).to(torch.float64).numpy()
    got = F.e8m0_to_float(np.arange(256))
    assert np.isnan(got[255]) and np.isnan(ref[255])
    assert np.array_equal(got[:255], ref[:255])


def test_e4m3_decode_all_codes_torch():
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = F.e4m3_to_float(np.arange(256))
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got)) and nan.sum() == 2     # 0x7F and 0xFF
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.nanmax(got) == 448.0 and np.nanmin(got) == -448.0
    assert got[1] == 2.0 ** -9                                        # smallest subnormal


def _e4m3_finite_values():
    v = F.e4m3_to_float(np.arange(128))
    return np.unique(v[~np.isnan(v)])          # 0 .. 448, ascending


def test_e4m3_encode_midpoints_and_neighbours():
    """Every midpoint between adjacent E4M3 values, +-1 float32 ulp, and the values
    themselves: compared with torch's round-to-nearest-even cast (in range)."""
    vals = _e4m3_finite_values()
    mids = ((vals[:-1] + vals[1:]) / 2).astype(np.float32)
    probes = np.concatenate([vals.astype(np.float32), mids,
                             np.nextafter(mids, np.float32(np.inf)),
                             np.nextafter(mids, np.float32(-np.inf))])
    probes = np.concatenate([probes, -probes])
    ref = torch.from_numpy(probes).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = F.float_to_e4m3_rne_sat(probes)
    assert np.array_equal(got, ref)


def test_e4m3_encode_random_and_saturation():
    rng = np.random.default_rng(7)
    x = (rng.standard_normal(200_000) * np.exp(rng.uniform(-9, 7, 200_000))).astype(np.float32)
    got = F.float_to_e4m3_rne_sat(x)
    inr = np.abs(x) <= 448
    ref = torch.from_numpy(x[inr]).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(got[inr], ref)
    # saturation: beyond 448 the code is +-448 (0x7E / 0xFE), never NaN
    big = np.array([448.5, 464.0, 479.9, 1e6, 3e38], dtype=np.float32)
    assert np.all(F.float_to_e4m3_rne_sat(big) == 0x7E)
    assert np.all(F.float_to_e4m3_rne_sat(-big) == 0xFE)
    # signed zeros and underflow keep the sign
    tiny = np.array([0.0, -0.0, 2.0 ** -11, -(2.0 ** -11)], dtype=np.float32)
    assert list(F.float_to_e4m3_rne_sat(tiny)) == [0x00, 0x80, 0x00, 0x80]


def test_bf16_rne_torch():
    rng = np.random.default_rng(3)
    x = (rng.standard_normal(100_000) * 10.0 ** rng.uniform(-5, 5, 100_000)).astype(np.float32)
    u = rng.integers(0, 2 ** 16, 1000, dtype=np.uint32)
    ties = ((u << 16) | 0x8000).view(np.float32)           # exact bf16 ties
    x = np.concatenate([x, ties[np.isfinite(ties)]])
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(F.f32_to_bf16_bits(x), ref)
    assert np.array_equal(F.bf16_bits_to_float(ref),
                          torch.from_numpy(ref.view(np.int16)).view(torch.bfloat16).float().numpy())


def test_round_f64_to_bf16_brute_force():
    """Nearest bf16 by enumerating the two bf16 neighbours (exact in float64)."""
    rng = np.random.default_rng(11)
    v = rng.standard_normal(20_000) * 10.0 ** rng.uniform(-3, 4, 20_000)
    got = F.round_f64_to_bf16(v).astype(np.float64)
    for x, g in zip(v[:4000], got[:4000]):
        b = int(F.f32_to_bf16_bits(np.float32(x)))         # a neighbour (+-1 step)
        cands = [F.bf16_bits_to_float(np.uint16((b + d) & 0xFFFF)).astype(np.float64)
                 for d in (-1, 0, 1)]
        cands = [c for c in cands if np.isfinite(c) and np.sign(c) == np.sign(x)]
        dist = [abs(c - x) for c in cands]
        best = min(dist)
        winners = [c for c, d in zip(cands, dist) if d == best]
        if len(winners) == 2:   # tie: even mantissa
            winners = [c for c in winners if int(F.f32_to_bf16_bits(np.float32(c))) % 2 == 0]
        assert g == winners[0]


def test_quantizer_invariants():
    rng = np.random.default_rng(5)
    v = (rng.standard_normal((64, 2560)) * rng.uniform(0.01, 100, (64, 1))).astype(np.float32)
    codes, scale = F.quantize_fp8_lastdim(v)
    dec = F.e4m3_to_float(codes) * scale[:, None].astype(np.float64)
    # the element of largest magnitude maps to +-448 exactly (its quotient is 448 to 1 ulp)
    imax = np.argmax(np.abs(v), axis=1)
    assert np.all(np.abs(F.e4m3_to_float(codes[np.arange(64), imax])) == 448.0)
    # error bound: half an E4M3 step (relative 2^-4 in the normal range, 2^-10 absolute below)
    t = np.abs(v.astype(np.float64) / scale[:, None])
    bound = np.where(t >= 2.0 ** -6, t * 2.0 ** -4, 2.0 ** -10) * scale[:, None] * (1 + 1e-6)
    assert np.all(np.abs(dec - v) <= bound + 1e-30)
    # zero vector: scale 1, zero codes
    c0, s0 = F.quantize_fp8_lastdim(np.zeros((1, 32), np.float32))
    assert s0[0] == 1.0 and not c0.any()


def test_quantizer_matches_torch_route():
    """Same steps done with torch float32 ops and torch's E4M3 cast."""
    rng = np.random.default_rng(9)
    v = (rng.standard_normal((32, 2560)) * 3).astype(np.float32)
    codes, scale = F.quantize_fp8_lastdim(v)
    tv = torch.from_numpy(v)
    ts = tv.abs().amax(dim=1) / torch.tensor(448.0)
    tq = (tv / ts[:, None]).clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ts.numpy(), scale)
    assert np.array_equal(tq, codes)
