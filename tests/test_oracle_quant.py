"""Pins of the oracle's MXFP4 and FP8 per-row quantizers.

MXFP4: "Kimi-K3 DSpark O-Proj-only MXFP4", "Exact quantization coverage" (E2M1
codes, E8M0 scale, 32 consecutive input channels per scale; stored weight
(7168, 8192), scale (7168, 256)); shared-exponent rule of OCP MX v1.0.
FP8: "Kimi-K3-DSpark-FP8-PTPC", "Phase 1 FP8 PTPC Quantization" (E4M3,
per-output-channel FP32 (out, 1) scale, dynamic per-token activations).
"""
import math
import struct
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
import synth
from conftest import read_golden


def f32_to_bf16_bits(v):
    """Exact only for values representable in bf16 (asserted)."""
    u = struct.unpack("<I", struct.pack("<f", v))[0]
    assert u & 0xFFFF == 0, v
    return u >> 16


def bits_to_float(b):
    return struct.unpack("<f", struct.pack("<I", (int(b) & 0xFFFF) << 16))[0]


# ---------------------------------------------------------------- MX block
def test_mx_single_one():
    x = np.zeros(32, np.uint16)
    x[5] = 0x3F80  # 1.0
    codes, sc = oracle.mx_quantize_block(x)
    assert sc == 125  # floor(log2 1) - 2 = -2 -> 125
    assert codes[5] == 0x6  # 1 * 2^2 = 4 -> code 6
    assert (np.delete(codes, 5) == 0).all()


def test_mx_zero_block_and_signed_zero():
    x = np.zeros(32, np.uint16)
    x[3] = 0x8000  # -0.0
    codes, sc = oracle.mx_quantize_block(x)
    assert sc == 0
    assert codes[3] == 0x8 and (np.delete(codes, 3) == 0).all()


@pytest.mark.parametrize("bad", [0x7FC0, 0x7F80, 0xFF80])
def test_mx_nonfinite_block(bad):
    x = np.full(32, 0x3F80, np.uint16)
    x[7] = bad
    codes, sc = oracle.mx_quantize_block(x)
    assert sc == 0xFF and (codes == 0).all()


def _mx_block_exact(vals):
    """Independent statement with exact rationals: find e with
    2^(e+2) <= amax < 2^(e+3), clamp to [-127, 127], then round each x*2^-e
    to the E2M1 grid by an explicit nearest/tie-even search."""
    fr = [Fraction(v) for v in vals]
    amax = max(abs(v) for v in fr)
    if amax == 0:
        e = -127
    else:
        e = 0
        while Fraction(2) ** (e + 2) > amax:
            e -= 1
        while Fraction(2) ** (e + 3) <= amax:
            e += 1
        e = max(-127, min(127, e))
    grid = [Fraction(x) for x in (0, 0.5, 1, 1.5, 2, 3, 4, 6)]
    codes = []
    for v, raw in zip(fr, vals):
        t = abs(v) / Fraction(2) ** e
        d = [abs(t - g) for g in grid]
        best = min(d)
        cands = [i for i, di in enumerate(d) if di == best]
        c = cands[0] if len(cands) == 1 else [i for i in cands if i % 2 == 0][0]
        codes.append(c | (8 if math.copysign(1.0, raw) < 0 else 0))
    return codes, e + 127


def test_mx_block_vs_exact_rationals_random():
    rng = np.random.default_rng(1234)
    for trial in range(300):
        scale = 2.0 ** rng.integers(-130, 120)
        vals = rng.standard_normal(32) * scale
        if trial % 5 == 0:
            vals[rng.integers(0, 32)] *= 50
        bits = np.array([f32_to_bf16_bits(float(np.float32(torch.tensor(v, dtype=torch.float32)
                                                              .to(torch.bfloat16).float())))
                         for v in vals], np.uint16)
        fvals = [bits_to_float(b) for b in bits]
        want_codes, want_sc = _mx_block_exact(fvals)
        codes, sc = oracle.mx_quantize_block(bits)
        assert sc == want_sc
        assert codes.tolist() == want_codes


def test_mx_block_edge_values_vs_exact():
    x = synth.special_values_bf16().view(torch.int16).numpy().view(np.uint16).copy()
    fvals = [bits_to_float(b) for b in x]
    want_codes, want_sc = _mx_block_exact(fvals)
    codes, sc = oracle.mx_quantize_block(x)
    assert sc == want_sc and codes.tolist() == want_codes
    # a block of subnormals only: amax subnormal -> e clamps to -127
    sub = np.array([0x0040, 0x8020, 0x0001] + [0] * 29, np.uint16)
    codes, sc = oracle.mx_quantize_block(sub)
    assert sc == 0
    assert codes[:3].tolist() == _mx_block_exact([bits_to_float(b) for b in sub])[0][:3]
    assert codes[0] == 0x2  # 2^-127 * 2^127 = 1.0


def test_mx_roundtrip_dequant_requant():
    rng = np.random.default_rng(7)
    for _ in range(200):
        codes = rng.integers(0, 16, 32).astype(np.uint8)
        codes[rng.integers(0, 32)] = rng.choice([6, 7, 14, 15])  # max magnitude 4 or 6
        sc = int(rng.integers(2, 253))
        vals = [oracle.e2m1_value(int(c)) * oracle.e8m0_value(sc) for c in codes]
        bits = np.array([f32_to_bf16_bits(v) for v in vals], np.uint16)
        c2, s2 = oracle.mx_quantize_block(bits)
        assert s2 == sc and (c2 == codes).all()


def test_mx_max_lands_on_4_or_6():
    rng = np.random.default_rng(99)
    x = synth.bf16_randn(64, 32 * 16, seed=5, outlier_frac=0.01)
    codes, sf = oracle.mx_quantize_rows(x)
    xf = x.float().numpy().reshape(64, 16, 32)
    unpacked = np.stack([codes & 0xF, codes >> 4], -1).reshape(64, 16, 32)
    imax = np.abs(xf).argmax(-1)
    mags = np.take_along_axis(unpacked, imax[..., None], -1)[..., 0] & 7
    assert set(np.unique(mags).tolist()) <= {6, 7}


def test_mx_scale_invariance_power_of_two():
    x = synth.bf16_randn(8, 256, seed=11, outlier_frac=0.01)
    c0, s0 = oracle.mx_quantize_rows(x)
    for j in (-20, -3, 1, 17):
        xs = (x.float() * 2.0 ** j).to(torch.bfloat16)  # exact power-of-two scaling
        c1, s1 = oracle.mx_quantize_rows(xs)
        assert (c1 == c0).all()
        assert (s1.astype(int) == s0.astype(int) + j).all()


def test_mx_rows_packing_low_nibble_is_lower_k():
    x = torch.zeros(1, 64, dtype=torch.bfloat16)
    x[0, 0] = 1.0      # code 6 at k=0  (scale of block 0 set by this element)
    x[0, 1] = -0.5     # -0.5 * 4 = -2 -> code 0xC at k=1
    x[0, 32] = 3.0     # block 1: e = -1, 3 * 2 = 6 -> code 7 at k=32
    codes, sf = oracle.mx_quantize_rows(x)
    assert codes.shape == (1, 32) and sf.shape == (1, 2)
    assert codes[0, 0] == (0x6 | (0xC << 4))
    assert codes[0, 16] == 0x7
    assert sf[0].tolist() == [125, 126]


def test_mx_rows_match_block_function():
    x = synth.activation(3, 256, seed=3)
    codes, sf = oracle.mx_quantize_rows(x)
    xb = x.view(torch.int16).numpy().view(np.uint16)
    for r in range(3):
        for g in range(8):
            c32, sc = oracle.mx_quantize_block(np.ascontiguousarray(xb[r, g * 32:(g + 1) * 32]))
            assert sf[r, g] == sc
            packed = (c32[0::2] | (c32[1::2] << 4)).astype(np.uint8)
            assert (codes[r, g * 16:(g + 1) * 16] == packed).all()


# ---------------------------------------------------------------- byte accounting
def test_byte_accounting_matches_checkpoint_sizes():
    g = {k: v for k, v in read_golden("checkpoint_bytes.txt")[1:]}
    N, K, L = int(g["N"]), int(g["K"]), int(g["layers"])
    # shapes produced by the oracle on a reduced row count, scaled to N rows
    x = synth.weight(4, K, seed=0)
    codes, sf = oracle.mx_quantize_rows(x)
    assert codes.shape == (4, K // 2) and sf.shape == (4, int(g["scale_cols"]))
    mx_bytes = N * codes.shape[1] + N * sf.shape[1]
    q, s = oracle.fp8_quantize_rows(x)
    fp8_bytes = N * q.shape[1] + N * s.dtype.itemsize
    assert mx_bytes == 31_195_136 and fp8_bytes == 58_748_928
    delta_gib = L * (fp8_bytes - mx_bytes) / 2 ** 30
    printed = float(g["fp8_gib"]) - float(g["mxfp4_gib"])
    assert abs(delta_gib - printed) <= 2 * float(g["printed_precision_gib"])
    # a 2-byte or 8-bit element code, or a scale per 16, would miss by far
    assert abs(L * (fp8_bytes - (N * K + N * K // 32)) / 2 ** 30 - printed) > 0.05


# ---------------------------------------------------------------- swizzle
def test_sf_swizzle_is_bijection():
    for rows, G in [(1, 4), (130, 8), (256, 256), (7168, 256)]:
        r = np.repeat(np.arange(rows), G)
        g = np.tile(np.arange(G), rows)
        off = np.array([oracle.sf_swizzled_offset(int(a), int(b), G) for a, b in
                        zip(r[:: max(1, len(r) // 5000)], g[:: max(1, len(r) // 5000)])])
        assert off.max() < oracle.sf_swizzled_bytes(rows, G)
    rows, G = 300, 8
    sf = np.arange(rows * G, dtype=np.int64).reshape(rows, G).astype(np.uint8)
    swz = oracle.sf_swizzle(sf, pad_value=0)
    assert len(swz) == 384 * G
    allo = [oracle.sf_swizzled_offset(r, g, G) for r in range(384) for g in range(G)]
    assert sorted(allo) == list(range(384 * G))
    assert (oracle.sf_unswizzle(swz, rows, G) == sf).all()


# ---------------------------------------------------------------- FP8 rows
def test_fp8_row_with_amax_448_has_unit_scale():
    x = synth.bf16_randn(4, 512, seed=21)
    xf = x.float()
    xf[:, 7] = 448.0
    xf = xf.clamp(-448, 448).to(torch.bfloat16)
    q, s = oracle.fp8_quantize_rows(xf)
    assert (s == 1.0).all()
    want = xf.float().to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert (q == want).all()


def test_fp8_power_of_two_invariance():
    x = synth.activation(6, 1024, seed=22)
    q0, s0 = oracle.fp8_quantize_rows(x)
    for j in (-9, 4):
        q1, s1 = oracle.fp8_quantize_rows((x.float() * 2.0 ** j).to(torch.bfloat16))
        assert (q1 == q0).all()
        assert (s1 == s0 * np.float32(2.0 ** j)).all()


def test_fp8_matches_library_division_and_cast():
    x = synth.activation(16, 2048, seed=23)
    q, s = oracle.fp8_quantize_rows(x)
    xf = x.float().numpy()
    amax = np.abs(xf).max(1).astype(np.float32)
    s_ref = amax / np.float32(448.0)  # numpy binary32 division
    assert (s == s_ref).all()
    t = (xf / s_ref[:, None]).astype(np.float32)
    want = torch.from_numpy(t).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert (q == want).all()


def test_fp8_zero_and_nonfinite_rows():
    x = torch.zeros(3, 64, dtype=torch.bfloat16)
    x[0, 5] = -0.0
    x[1, 3] = float("nan")
    x[2, 9] = float("inf")
    q, s = oracle.fp8_quantize_rows(x)
    assert s[0] == 1.0 and q[0, 5] == 0x80 and (np.delete(q[0], 5) == 0).all()
    assert math.isnan(s[1]) and math.isnan(s[2])
    assert (q[1:] == 0).all()
