"""Pins of the oracle's grouped (MoE) A4W4 GEMM ("Kimi-K3-Quark-MXFP4-
AttnFP8", "Model Overview": the experts are OCP MXFP4): every token row goes
through the weight of the expert whose group it is in, and through no other.
"""
import numpy as np
import pytest

import oracle


def pack(c):
    return (c[:, 0::2] | (c[:, 1::2] << 4)).astype(np.uint8)


def test_rows_only_see_their_own_expert():
    """Expert e's weight holds 1.0 at column e of every output row, and a
    token row of group e holds 1.0 at column e only (unit scales, code 127).
    Through its own expert every row gives 1.0 in every output; through any
    other expert it would give 0, which the rotated assignment checks."""
    E, N, K = 4, 8, 64
    off = [0, 3, 3, 7, 9]  # group 1 empty
    M = off[-1]
    w_codes, w_sf = [], []
    for e in range(E):
        w = np.zeros((N, K), np.uint8)
        w[:, e] = 0x2  # 1.0
        w_codes.append(pack(w))
        w_sf.append(np.full((N, K // 32), 127, np.uint8))
    a = np.zeros((M, K), np.uint8)
    for e in range(E):
        a[off[e]:off[e + 1], e] = 0x2
    ref, bound = oracle.gemm_a4w4_grouped(pack(a), np.full((M, K // 32), 127, np.uint8), w_codes, w_sf, off)
    assert (ref == 1.0).all() and (bound == 1.0).all()
    # the same rows against a rotated expert assignment see nothing
    ref2, _ = oracle.gemm_a4w4_grouped(pack(a), np.full((M, K // 32), 127, np.uint8),
                                       w_codes[1:] + w_codes[:1], w_sf, off)
    assert (ref2 == 0.0).all()


def test_one_group_is_the_plain_gemm_and_empty_groups_are_allowed():
    rng = np.random.default_rng(0)
    M, N, K = 5, 16, 96
    a = rng.integers(0, 16, (M, K)).astype(np.uint8)
    w = rng.integers(0, 16, (N, K)).astype(np.uint8)
    asf = rng.integers(120, 135, (M, K // 32)).astype(np.uint8)
    wsf = rng.integers(120, 135, (N, K // 32)).astype(np.uint8)
    ref, bound = oracle.gemm_a4w4(pack(a), asf, pack(w), wsf)
    g_ref, g_bound = oracle.gemm_a4w4_grouped(pack(a), asf, [pack(w), pack(w)], [wsf, wsf], [0, 0, M])
    assert (g_ref == ref).all() and (g_bound == bound).all()
    z_ref, _ = oracle.gemm_a4w4_grouped(pack(a)[:0], asf[:0], [pack(w)], [wsf], [0, 0])
    assert z_ref.shape == (0, N)


def test_groups_must_tile_the_rows():
    a = np.zeros((4, 16), np.uint8)
    w = [np.zeros((8, 16), np.uint8)]
    s = [np.zeros((8, 1), np.uint8)]
    with pytest.raises(AssertionError):
        oracle.gemm_a4w4_grouped(a, np.zeros((4, 1), np.uint8), w, s, [0, 3])
