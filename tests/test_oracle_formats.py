"""Pins of the oracle's number formats against library routines and closed forms.

E4M3 and bf16 are checked against torch's own float8_e4m3fn / bfloat16 types
(an independent implementation); UE8M0 and exp against their definitions.
"""
import math

import numpy as np
import pytest
import torch

import oracle


def test_e4m3_decode_matches_torch_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_to_f64(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert nan.sum() == 2  # 0x7f and 0xff
    assert np.array_equal(ours[~nan], ref[~nan])
    assert ours[0x7E] == 448.0 and ours[0x01] == 2.0 ** -9


def test_e4m3_roundtrip_every_code():
    codes = np.arange(256, dtype=np.uint8)
    keep = (codes & 0x7F) != 0x7F
    vals = oracle.e4m3_to_f64(codes[keep]).astype(np.float32)
    back = oracle.f32_to_e4m3(vals)
    assert np.array_equal(back, codes[keep])


def test_e4m3_ties_to_even_and_saturation():
    pos = oracle.e4m3_to_f64(np.arange(0x7F, dtype=np.uint8))
    mids = ((pos[:-1] + pos[1:]) / 2).astype(np.float32)
    assert np.array_equal(mids.astype(np.float64), (pos[:-1] + pos[1:]) / 2)  # exact in fp32
    got = oracle.f32_to_e4m3(mids)
    lo = np.arange(0x7E, dtype=np.uint8)
    expect = np.where(lo % 2 == 0, lo, lo + 1).astype(np.uint8)
    assert np.array_equal(got, expect)
    sat = oracle.f32_to_e4m3(np.array([448.0, 449.0, 464.0, 500.0, 1e30, np.inf, -np.inf,
                                       -1e9], np.float32))
    assert list(sat) == [0x7E] * 6 + [0xFE] * 2


def test_e4m3_encode_matches_torch_in_range():
    g = np.random.default_rng(123)
    x = np.concatenate([g.normal(size=200000) * 10.0 ** g.uniform(-4, 2.5, size=200000),
                        g.uniform(-448, 448, size=50000)]).astype(np.float32)
    x = x[np.abs(x) <= 448]
    ours = oracle.f32_to_e4m3(x)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)


def test_bf16_matches_torch():
    g = np.random.default_rng(7)
    x = (g.normal(size=300000) * 10.0 ** g.uniform(-30, 30, size=300000)).astype(np.float32)
    # exact ties (low half 0x8000) with both parities of the kept half
    ties = (np.arange(0x3F800000, 0x3F800000 + 64 * 0x10000, 0x10000, dtype=np.uint32)
            + 0x8000).view(np.float32)
    x = np.concatenate([x, ties, np.array([0.0, -0.0, 3.4e38, -3.4e38, 1e-40], np.float32)])
    ours = oracle.f32_to_bf16(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    assert np.array_equal(oracle.bf16_to_f32(ours),
                          torch.from_numpy(ref.view(np.int16)).view(torch.bfloat16).float().numpy())


@pytest.mark.parametrize("amax", [1e-30, 3e-5, 0.01, 0.5, 1.0, 447.9, 448.0, 448.1, 896.0, 1e6,
                                  3.3e38])
def test_ue8m0_is_smallest_nonsaturating_power(amax):
    e = oracle.ue8m0_exponent(amax)
    a = float(np.float32(amax))
    assert a <= 448.0 * 2.0 ** e
    assert a > 448.0 * 2.0 ** (e - 1)


def test_ue8m0_exact_powers_and_zero():
    for k in range(-20, 20):
        assert oracle.ue8m0_exponent(448.0 * 2.0 ** k) == k
    assert oracle.ue8m0_exponent(0.0) == 0


def test_expf_error_bound_against_libm():
    xs = np.concatenate([np.linspace(-87, 0, 200001), -np.logspace(-8, 1.9, 2000)]).astype(np.float32)
    worst = 0.0
    for x in xs[::7]:
        ours = oracle.expf(float(x))
        ref = math.exp(float(x))
        worst = max(worst, abs(ours - ref) / ref)
    # 2^-23 is one fp32 ulp at 1.0; Horner without FMA plus the Cody-Waite split
    # stays within a few ulp
    assert worst < 4 * 2.0 ** -23, worst
    assert oracle.expf(0.0) == 1.0
    assert oracle.expf(-88.0) == 0.0


def test_expf_monotone():
    xs = np.linspace(-20, 0, 40001).astype(np.float32)
    ys = np.array([oracle.expf(float(x)) for x in xs])
    assert np.all(np.diff(ys) >= 0)
