"""Pins of the oracle's element formats against what the standards fix.

E2M1 and E8M0 are the OCP MX v1.0 encodings the pages name ("MXFP4 E2M1",
"E8M0" in "Kimi-K3 DSpark O-Proj-only MXFP4", "Exact quantization coverage";
"OCP MXFP4" in "Kimi-K3-Quark-MXFP4-AttnFP8", "Model Overview").  E4M3 is
torch.float8_e4m3fn ("Kimi-K3-DSpark-FP8-PTPC", "Phase 1 FP8 PTPC
Quantization"), so torch's own cast is an independent library check for
in-range values.
"""
import math
import struct
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from conftest import read_golden


def bf16_bits_to_float(b):
    return struct.unpack("<f", struct.pack("<I", (b & 0xFFFF) << 16))[0]


def test_bf16_widening_is_bit_shift():
    for b in [0x0000, 0x8000, 0x3F80, 0xBF80, 0x0001, 0x7F7F, 0x4049, 0x3C23]:
        assert oracle.bf16_to_f32(b) == bf16_bits_to_float(b)
        assert math.copysign(1, oracle.bf16_to_f32(b)) == math.copysign(1, bf16_bits_to_float(b))


def test_e2m1_decode_table():
    for code, val in read_golden("e2m1_values.txt"):
        got = oracle.e2m1_value(int(code))
        assert got == float(val)
        assert math.copysign(1.0, got) == math.copysign(1.0, float(val))


def test_e2m1_decode_from_bit_fields():
    # independent of the oracle's table: (-1)^s * 2^(E-1) * (1 + m/2), E>0;
    # subnormal E=0: (-1)^s * m/2
    for code in range(16):
        s, E, m = code >> 3, (code >> 1) & 3, code & 1
        mag = Fraction(m, 2) if E == 0 else Fraction(2) ** (E - 1) * (1 + Fraction(m, 2))
        v = oracle.e2m1_value(code)
        assert Fraction(abs(v)) == mag
        assert (math.copysign(1.0, v) < 0) == bool(s)


def test_e8m0_points():
    for code, lg in read_golden("e8m0_points.txt"):
        v = oracle.e8m0_value(int(code))
        if lg == "nan":
            assert math.isnan(v)
        else:
            assert v == 2.0 ** int(lg)


def test_e8m0_all_codes():
    for c in range(255):
        assert oracle.e8m0_value(c) == math.ldexp(1.0, c - 127)


def _e2m1_rne_exact(v: Fraction) -> int:
    """Independent rule: the spacing of the E2M1 grid is 1/2 below 2, 1 in
    [2, 4), 2 from 4 on; round |v| to a multiple of the spacing with ties to
    an even multiple, saturate at 6, map the value back to its code."""
    a = abs(v)
    step = Fraction(1, 2) if a < 2 else (Fraction(1) if a < 4 else Fraction(2))
    q = a / step
    lo = math.floor(q)
    frac = q - lo
    n = lo + 1 if frac > Fraction(1, 2) or (frac == Fraction(1, 2) and lo % 2 == 1) else lo
    r = min(n * step, Fraction(6))
    return [Fraction(x) for x in (0, 0.5, 1, 1.5, 2, 3, 4, 6)].index(r)


def test_e2m1_rounding_golden_ties():
    for mag, code in read_golden("e2m1_ties.txt"):
        assert oracle.e2m1_round(float(mag)) == int(code)
        assert oracle.e2m1_round(-float(mag)) == int(code) | 8


def test_e2m1_roundtrip_all_codes():
    for code in range(16):
        assert oracle.e2m1_round(oracle.e2m1_value(code)) == code


def test_e2m1_rounding_exhaustive_bf16():
    # every non-negative bf16 value below 8 (and its negation)
    for b in range(0x0000, 0x4100):
        f = bf16_bits_to_float(b)
        want = _e2m1_rne_exact(Fraction(f))
        assert oracle.e2m1_round(f) == want, (hex(b), f)
        assert oracle.e2m1_round(-f) == want | 8, (hex(b), f)


def test_e4m3_decode_matches_torch():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for c in range(256):
        got = oracle.e4m3_value(c)
        if math.isnan(ref[c]):
            assert math.isnan(got), c
        else:
            assert got == ref[c], c
    assert oracle.e4m3_value(0x7E) == 448.0
    assert oracle.e4m3_value(0x01) == 2.0 ** -9


def test_e4m3_rounding_vs_torch_all_inrange_bf16():
    bits = np.arange(0, 0x8000, dtype=np.uint32)
    vals = (bits << 16).view(np.float32)
    keep = np.isfinite(vals) & (np.abs(vals) <= 448.0)
    vals = vals[keep]
    want = torch.from_numpy(vals.copy()).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    for v, w in zip(vals.tolist(), want.tolist()):
        assert oracle.e4m3_round(v) == w, v
        assert oracle.e4m3_round(-v) == (w | 0x80), v


def test_e4m3_saturation_and_signed_zero():
    assert oracle.e4m3_round(1.0e6) == 0x7E
    assert oracle.e4m3_round(-1.0e6) == 0xFE
    assert oracle.e4m3_round(480.0) == 0x7E
    assert oracle.e4m3_round(-0.0) == 0x80
    assert oracle.e4m3_round(-1e-9) == 0x80
    assert oracle.e4m3_round(2.0 ** -10) == 0x00  # tie to even (0)
    assert oracle.e4m3_round(3 * 2.0 ** -10) == 0x02  # tie between 1 and 2 -> 2


def test_floor_log2_exact():
    for e in range(-149, 128):
        a = math.ldexp(1.0, e)
        if e >= -149:
            assert oracle.floor_log2(a) == e
    assert oracle.floor_log2(3.0) == 1
    assert oracle.floor_log2(0.75) == -1
    assert oracle.floor_log2(np.float32(2.0 ** -130 * 1.9)) == -130
