"""Pins for the oracle's number codecs (e4m3, bf16, ue8m0).

Each codec is checked against something other than itself: the format's
closed form, fixtures worked from the published definitions
(tests/golden/), and PyTorch's own CPU dtype casts used as a library.
"""
import math
import os
import struct

import numpy as np
import pytest
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_fixture(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                rows.append(line.split())
    return rows


def test_e4m3_decode_golden(orc):
    for code_hex, val in _read_fixture("e4m3_codes.txt"):
        got = orc.e4m3_decode(np.array([int(code_hex, 16)], np.uint8))[0]
        if val == "nan":
            assert math.isnan(got)
        else:
            assert got == float(val) and math.copysign(1, got) == math.copysign(1, float(val))


def test_e4m3_decode_all_codes_vs_torch(orc):
    codes = np.arange(256, dtype=np.uint8)
    ours = orc.e4m3_decode(codes)
    lib = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(lib)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], lib[~nan])
    assert np.array_equal(np.signbit(ours[~nan]), np.signbit(lib[~nan]))
    assert nan.sum() == 2


def _e4m3_probe_values():
    codes = np.arange(0, 0x7F, dtype=np.uint8)
    vals = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    mids = (vals[:-1] + vals[1:]) / 2          # exact ties
    f32 = np.concatenate([vals, mids]).astype(np.float32)
    up = np.nextafter(f32, np.float32(np.inf))
    dn = np.nextafter(f32, np.float32(-np.inf))
    rng = np.random.default_rng(0)
    rnd = np.concatenate([rng.standard_normal(20000) * s for s in (1e-3, 0.05, 1, 30, 200)])
    allv = np.concatenate([f32, up, dn, rnd.astype(np.float32)])
    allv = allv[np.abs(allv) <= 464.0]
    return np.concatenate([allv, -allv]).astype(np.float32)


def test_e4m3_encode_vs_torch_cast(orc):
    v = _e4m3_probe_values()
    ours = orc.e4m3_encode(v)
    lib = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    # Signed zeros: compare values, then signs only where nonzero.
    assert np.array_equal(orc.e4m3_decode(ours), orc.e4m3_decode(lib))


def test_e4m3_encode_ties_to_even_and_saturation(orc):
    # 1.0625 lies halfway between 1.0 (0x38, even) and 1.125 (0x39, odd).
    assert orc.e4m3_encode(np.array([1.0625], np.float32))[0] == 0x38
    # 1.1875 halfway between 1.125 (0x39) and 1.25 (0x3A, even).
    assert orc.e4m3_encode(np.array([1.1875], np.float32))[0] == 0x3A
    # Saturating: everything finite beyond 448 becomes +-448, never NaN.
    big = np.array([448.0, 449.0, 464.0, 470.0, 480.0, 1e6, 3e38], np.float32)
    assert (orc.e4m3_encode(big) == 0x7E).all()
    assert (orc.e4m3_encode(-big) == 0xFE).all()
    # Half the smallest subnormal rounds to zero (tie, even); just above rounds up.
    assert orc.e4m3_encode(np.array([2.0 ** -10], np.float32))[0] == 0x00
    assert orc.e4m3_encode(np.array([np.nextafter(np.float32(2.0 ** -10), np.float32(1))], np.float32))[0] == 0x01
    assert orc.e4m3_encode(np.array([np.nan], np.float32))[0] in (0x7F, 0xFF)


def test_bf16_encode_vs_torch_on_float32(orc):
    rng = np.random.default_rng(1)
    v = np.concatenate([rng.standard_normal(200000) * s for s in (1e-30, 1e-3, 1, 1e3, 1e30)])
    v = v.astype(np.float32)
    # add exact bf16 ties: a bf16 value plus half its ulp
    base = torch.from_numpy(rng.standard_normal(5000).astype(np.float32)).to(torch.bfloat16).to(torch.float32).numpy()
    bits = base.view(np.uint32)
    ties = ((bits & 0xFFFF0000) | 0x8000).view(np.float32)
    v = np.concatenate([v, ties, np.float32([0.0, -0.0, 1e-45, 3.3e38, 3.4e38])])
    ours = orc.bf16_encode(v.astype(np.float64))
    lib = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, lib)


def test_bf16_encode_single_rounding_from_double(orc):
    # 1 + 2^-8 + 2^-40 is above the tie between 1 and 1+2^-7: one rounding
    # from double goes up; a detour through float32 would round to the tie and
    # then to even (1.0).
    v = 1.0 + 2.0 ** -8 + 2.0 ** -40
    assert orc.bf16_encode(np.array([v]))[0] == 0x3F81
    assert orc.bf16_encode(np.array([1.0 + 2.0 ** -8]))[0] == 0x3F80   # tie -> even
    assert orc.bf16_encode(np.array([1.0 + 3 * 2.0 ** -8]))[0] == 0x3F82  # tie -> even
    assert orc.bf16_encode(np.array([-2.5]))[0] == 0xC020


def test_ue8m0_golden_rule(orc):
    for bits_hex, byte, *_ in _read_fixture("ue8m0_rule.txt"):
        s = struct.unpack("<f", struct.pack("<I", int(bits_hex, 16)))[0]
        assert orc.ue8m0_encode(np.array([s], np.float32))[0] == int(byte), bits_hex


def test_ue8m0_is_power_of_two_ceiling_for_normals(orc):
    rng = np.random.default_rng(2)
    s = np.exp(rng.uniform(-80, 80, 100000)).astype(np.float32)
    s = np.concatenate([s, np.float32([2.0 ** k for k in range(-120, 120)])])
    b = orc.ue8m0_encode(s).astype(np.int64)
    for si, bi in zip(s[::97], b[::97]):
        m, e = math.frexp(float(si))           # si = m * 2^e, m in [0.5, 1)
        ceil_log2 = e - 1 if m == 0.5 else e
        assert bi == 127 + ceil_log2
    dec = np.array([orc.ue8m0_decode(x) for x in b[:2000]])
    assert (dec >= s[:2000]).all() and (dec / 2 < s[:2000]).all()
