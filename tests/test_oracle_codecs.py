"""Pins for the oracle's number formats (E4M3FN, bf16, E2M1, E8M0).

Each codec is checked against something other than itself: torch's own float8
and bfloat16 casts, exact rational rounding with ``fractions``, and the code
tables of the OCP FP8 and OCP MX v1.0 specifications (tests/golden/, cited).
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _table(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                a, b = line.split()
                rows.append((int(a, 16), float(b)))
    return rows


def _torch_e4m3_value(codes):
    return torch.tensor(codes, dtype=torch.uint8).view(torch.float8_e4m3fn).float().double().numpy()


def test_e4m3_decode_all_codes_match_torch(orc):
    codes = np.arange(256, dtype=np.uint8)
    ours = orc.e4m3_decode(codes)
    ref = _torch_e4m3_value(codes)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert nan.sum() == 2  # S.1111.111 only
    assert np.array_equal(ours[~nan], ref[~nan])
    # signed zero
    assert math.copysign(1.0, ours[0x80]) == -1.0


def test_e4m3_spec_table(orc):
    for code, value in _table("ocp_fp8_e4m3.txt"):
        got = float(orc.e4m3_decode(np.uint8(code)))
        assert got == value, (hex(code), got, value)
        if not (value == 0 and code == 0x80):
            assert int(orc.e4m3_encode(np.float32(value))) == code


def _e4m3_grid():
    v = orc_vals = _torch_e4m3_value(np.arange(256, dtype=np.uint8))
    g = np.unique(v[np.isfinite(v) & (v >= 0)])
    return g


def test_e4m3_encode_matches_torch_cast(orc):
    rng = np.random.default_rng(0)
    grid = _e4m3_grid()
    mids = (grid[:-1] + grid[1:]) / 2  # exact ties (all representable in fp32)
    parts = [
        rng.standard_normal(400_000).astype(np.float32) * np.float32(100.0),
        rng.standard_normal(200_000).astype(np.float32) * np.float32(0.01),  # subnormals
        (rng.random(200_000) * 448).astype(np.float32),
        mids.astype(np.float32), -mids.astype(np.float32),
        np.nextafter(mids.astype(np.float32), np.float32(np.inf)),
        np.nextafter(mids.astype(np.float32), np.float32(-np.inf)),
        grid.astype(np.float32), -grid.astype(np.float32),
    ]
    v = np.concatenate(parts)
    v = v[np.abs(v) <= 448]
    ours = orc.e4m3_encode(v)
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    bad = np.nonzero(ours != ref)[0]
    assert bad.size == 0, (v[bad[:5]], ours[bad[:5]], ref[bad[:5]])


def test_e4m3_encode_saturates(orc):
    # satfinite: everything beyond the largest finite value clamps to +-448
    v = np.array([448.0, 449.0, 463.9, 464.0, 480.0, 1e6, np.inf, -500.0, -np.inf], np.float32)
    out = orc.e4m3_encode(v)
    assert list(out) == [0x7E] * 7 + [0xFE] * 2


def test_e4m3_ties_round_to_even(orc):
    # 1.0625 lies halfway between 1.0 (mantissa 000) and 1.125 (mantissa 001)
    assert int(orc.e4m3_encode(np.float32(1.0625))) == 0x38
    # 1.1875 lies halfway between 1.125 (001) and 1.25 (010): even is 010
    assert int(orc.e4m3_encode(np.float32(1.1875))) == 0x3A
    # subnormal tie 1.5 * 2^-9 -> 2 * 2^-9
    assert int(orc.e4m3_encode(np.float32(1.5 * 2.0 ** -9))) == 0x02


def test_bf16_from_double_matches_torch_on_fp32_inputs(orc):
    rng = np.random.default_rng(1)
    v = np.concatenate([
        rng.standard_normal(300_000).astype(np.float32),
        (rng.standard_normal(100_000) * 1e30).astype(np.float32),
        (rng.standard_normal(100_000) * 1e-38).astype(np.float32),  # bf16 subnormals
    ])
    # exact ties: fp32 values whose low 16 bits are 0x8000
    ties = (rng.integers(0, 2**31, 50_000, dtype=np.uint32) & np.uint32(0x7F7F0000)) | np.uint32(0x8000)
    v = np.concatenate([v, ties.view(np.float32)])
    ours = orc.bf16_from_double(v.astype(np.float64))
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


def _bf16_exact_round(d: float) -> int:
    """Brute-force nearest-even bf16 of a double using exact rationals."""
    f = Fraction(d)
    sign = 0x8000 if f < 0 else 0
    a = abs(f)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    q = Fraction(2) ** (e - 7)
    n = a / q
    fl = n.numerator // n.denominator
    rem = n - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    val = fl * q
    e2 = e if val < Fraction(2) ** (e + 1) else e + 1
    m = int((val / Fraction(2) ** e2 - 1) * 128)
    return sign | ((e2 + 127) << 7) | m


def test_bf16_from_double_no_double_rounding(orc):
    rng = np.random.default_rng(2)
    # doubles just above a bf16 midpoint that first rounding to fp32 would pull
    # onto the midpoint (and then to even = down)
    base = rng.standard_normal(2000)
    bits = base.view(np.uint64) & np.uint64(0xFFFFE00000000000)
    mid = bits | np.uint64(1 << 44)  # exactly halfway in bf16 terms
    above = (mid + np.uint64(1)).view(np.float64)
    below = (mid - np.uint64(1)).view(np.float64)
    vals = np.concatenate([above, below, mid.view(np.float64), rng.standard_normal(2000) * 1e3])
    ours = orc.bf16_from_double(vals)
    ref = np.array([_bf16_exact_round(float(d)) for d in vals], dtype=np.uint16)
    assert np.array_equal(ours, ref)


def test_e2m1_spec_table(orc):
    rows = _table("ocp_mx_e2m1.txt")
    assert len(rows) == 16
    for nib, value in rows:
        got = float(orc.e2m1_decode(np.uint8(nib)))
        assert got == value and math.copysign(1, got) == math.copysign(1, value), (nib, got)


def test_e8m0(orc):
    s = np.arange(255, dtype=np.uint8)
    assert np.array_equal(orc.e8m0_decode(s), np.ldexp(1.0, s.astype(np.int64) - 127))
    assert math.isnan(float(orc.e8m0_decode(np.uint8(255))))
    assert float(orc.e8m0_decode(np.uint8(127))) == 1.0
