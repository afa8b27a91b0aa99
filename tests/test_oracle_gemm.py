"""Pins of the oracle's reference GEMMs (the Linear y = x . W^T over the
dequantized operands) against exact rational brute force and against a
plain integer matmul in the special case where every scale is 1.

A4W4: "Kimi-K3 DSpark O-Proj-only MXFP4", "Exact quantization coverage"
(MXFP4 operands, A4W4 dispatch).  PTPC: "Kimi-K3-DSpark-FP8-PTPC", "Phase 1
FP8 PTPC Quantization" (E4M3 weights with per-output-channel scales, dynamic
per-token activation scales).
"""
import math
from fractions import Fraction

import numpy as np
import pytest

import oracle


def e2m1_exact(code):
    s, E, m = code >> 3, (code >> 1) & 3, code & 1
    mag = Fraction(m, 2) if E == 0 else Fraction(2) ** (E - 1) * (1 + Fraction(m, 2))
    return -mag if s else mag


def e4m3_exact(code):
    s, E, m = code >> 7, (code >> 3) & 15, code & 7
    mag = Fraction(m, 8) * Fraction(2) ** -6 if E == 0 else (1 + Fraction(m, 8)) * Fraction(2) ** (E - 7)
    return -mag if s else mag


def unpack(codes):
    return np.stack([codes & 0xF, codes >> 4], -1).reshape(codes.shape[0], -1)


@pytest.mark.parametrize("M,N,K", [(1, 1, 32), (3, 4, 64), (4, 2, 128), (2, 3, 96)])
def test_a4w4_vs_exact_rational(M, N, K):
    rng = np.random.default_rng(M * 100 + N * 10 + K)
    a_codes = rng.integers(0, 256, (M, K // 2)).astype(np.uint8)
    w_codes = rng.integers(0, 256, (N, K // 2)).astype(np.uint8)
    a_sf = rng.integers(100, 150, (M, K // 32)).astype(np.uint8)
    w_sf = rng.integers(100, 150, (N, K // 32)).astype(np.uint8)
    ref, bound = oracle.gemm_a4w4(a_codes, a_sf, w_codes, w_sf)
    A, W = unpack(a_codes), unpack(w_codes)
    for m in range(M):
        for n in range(N):
            tot = Fraction(0)
            tot_abs = Fraction(0)
            for k in range(K):
                p = (e2m1_exact(int(A[m, k])) * Fraction(2) ** (int(a_sf[m, k // 32]) - 127)
                     * e2m1_exact(int(W[n, k])) * Fraction(2) ** (int(w_sf[n, k // 32]) - 127))
                tot += p
                tot_abs += abs(p)
            assert abs(Fraction(ref[m, n]) - tot) <= tot_abs * Fraction(1, 2 ** 50)
            assert Fraction(bound[m, n]) == tot_abs or abs(Fraction(bound[m, n]) - tot_abs) <= tot_abs * Fraction(1, 2 ** 50)


def test_a4w4_unit_scales_is_integer_matmul():
    # codes whose values are integers: 0, +-1, +-2, +-3, +-4, +-6
    int_codes = np.array([0, 2, 4, 5, 6, 7, 10, 12, 13, 14, 15], np.uint8)
    rng = np.random.default_rng(5)
    M, N, K = 5, 7, 256
    A = int_codes[rng.integers(0, len(int_codes), (M, K))]
    W = int_codes[rng.integers(0, len(int_codes), (N, K))]
    pack = lambda X: (X[:, 0::2] | (X[:, 1::2] << 4)).astype(np.uint8)
    sfa = np.full((M, K // 32), 127, np.uint8)
    sfw = np.full((N, K // 32), 127, np.uint8)
    ref, bound = oracle.gemm_a4w4(pack(A), sfa, pack(W), sfw)
    val = np.array([oracle.e2m1_value(int(c)) for c in range(16)]).astype(np.int64)
    Ai, Wi = val[A], val[W]
    assert (ref == (Ai @ Wi.T)).all()
    assert (bound == (np.abs(Ai) @ np.abs(Wi).T)).all()


def test_a4w4_row_subset_and_nan_scale():
    rng = np.random.default_rng(9)
    M, N, K = 6, 5, 64
    a = rng.integers(0, 256, (M, K // 2)).astype(np.uint8)
    w = rng.integers(0, 256, (N, K // 2)).astype(np.uint8)
    sa = rng.integers(120, 135, (M, 2)).astype(np.uint8)
    sw = rng.integers(120, 135, (N, 2)).astype(np.uint8)
    full, _ = oracle.gemm_a4w4(a, sa, w, sw)
    sub, _ = oracle.gemm_a4w4(a, sa, w, sw, rows=[4, 1])
    assert (sub == full[[4, 1]]).all()
    sa[2, 1] = 0xFF
    nanrow, _ = oracle.gemm_a4w4(a, sa, w, sw)
    assert np.isnan(nanrow[2]).all() and not np.isnan(nanrow[[0, 1, 3, 4, 5]]).any()


@pytest.mark.parametrize("M,N,K", [(1, 1, 32), (3, 4, 64), (4, 3, 128)])
def test_ptpc_vs_exact_rational(M, N, K):
    rng = np.random.default_rng(M + N + K)
    qa = rng.integers(0, 256, (M, K)).astype(np.uint8)
    qw = rng.integers(0, 256, (N, K)).astype(np.uint8)
    qa[(qa & 0x7F) == 0x7F] = 0x10  # no NaN codes
    qw[(qw & 0x7F) == 0x7F] = 0x21
    sa = (rng.random(M) * 3 + 0.01).astype(np.float32)
    sw = (rng.random(N) * 0.01 + 1e-4).astype(np.float32)
    ref, bound = oracle.gemm_ptpc(qa, sa, qw, sw)
    for m in range(M):
        for n in range(N):
            tot = sum(e4m3_exact(int(qa[m, k])) * e4m3_exact(int(qw[n, k])) for k in range(K))
            tot_abs = sum(abs(e4m3_exact(int(qa[m, k])) * e4m3_exact(int(qw[n, k]))) for k in range(K))
            want = tot * Fraction(float(sa[m])) * Fraction(float(sw[n]))
            want_abs = tot_abs * abs(Fraction(float(sa[m])) * Fraction(float(sw[n])))
            assert abs(Fraction(ref[m, n]) - want) <= want_abs * Fraction(1, 2 ** 50)
            assert abs(Fraction(bound[m, n]) - want_abs) <= want_abs * Fraction(1, 2 ** 50)


def test_ptpc_unit_scales_is_integer_matmul():
    # integer-valued E4M3 codes in [-16, 16]
    ints = [c for c in range(256) if (c & 0x7F) != 0x7F and
            float(oracle.e4m3_value(c)).is_integer() and abs(oracle.e4m3_value(c)) <= 16]
    ints = np.array(ints, np.uint8)
    rng = np.random.default_rng(3)
    M, N, K = 4, 6, 512
    qa = ints[rng.integers(0, len(ints), (M, K))]
    qw = ints[rng.integers(0, len(ints), (N, K))]
    ref, bound = oracle.gemm_ptpc(qa, np.ones(M, np.float32), qw, np.ones(N, np.float32))
    val = np.array([oracle.e4m3_value(c) if (c & 0x7F) != 0x7F else 0 for c in range(256)])
    Ai, Wi = val[qa].astype(np.int64), val[qw].astype(np.int64)
    assert (ref == Ai @ Wi.T).all()
    # swapping the roles of the operands transposes the result
    ref_t, _ = oracle.gemm_ptpc(qw, np.ones(N, np.float32), qa, np.ones(M, np.float32))
    assert (ref_t == ref.T).all()


def test_ptpc_scales_apply_per_token_and_per_channel():
    rng = np.random.default_rng(4)
    M, N, K = 3, 4, 64
    qa = rng.integers(0, 0x70, (M, K)).astype(np.uint8)
    qw = rng.integers(0, 0x70, (N, K)).astype(np.uint8)
    base, _ = oracle.gemm_ptpc(qa, np.ones(M, np.float32), qw, np.ones(N, np.float32))
    sa = np.array([2.0, 0.5, 8.0], np.float32)
    sw = np.array([1.0, 4.0, 0.25, 2.0], np.float32)
    got, _ = oracle.gemm_ptpc(qa, sa, qw, sw)
    assert (got == base * sa[:, None] * sw[None, :]).all()
