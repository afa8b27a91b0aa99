"""Helpers for the GPU parity tests: device handles, oracle comparisons."""
import numpy as np
import pytest
import torch

import oracle

# Tolerance for GEMM outputs (fp32 before the bf16 cast): the stated bound
# |gpu - oracle| <= 1e-5 * sum_k |a_k w_k| per element.
GEMM_REL_TOL = 1e-5


def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda", 0)


def np_u8(t):
    return t.detach().cpu().numpy().astype(np.uint8)


def assert_codes_equal(got, want, what):
    got = np.asarray(got)
    want = np.asarray(want)
    assert got.shape == want.shape, (what, got.shape, want.shape)
    bad = np.argwhere(got != want)
    assert bad.size == 0, f"{what}: {len(bad)} mismatches, first at {bad[:5].tolist()}: " \
                          f"got {got[tuple(bad[0])]} want {want[tuple(bad[0])]}"


def assert_gemm_close(y, ref, bound, what, tol=GEMM_REL_TOL):
    y = np.asarray(y, dtype=np.float64)
    assert y.shape == ref.shape, (what, y.shape, ref.shape)
    nan_ref = np.isnan(ref)
    assert (np.isnan(y) == nan_ref).all(), f"{what}: NaN pattern differs"
    err = np.abs(y - ref)
    ok = np.where(nan_ref, True, err <= tol * bound)
    if not ok.all():
        idx = np.argwhere(~ok)[:5]
        i0 = tuple(idx[0])
        raise AssertionError(f"{what}: {int((~ok).sum())} elements outside tolerance; first {idx.tolist()}"
                             f" got {y[i0]!r} ref {ref[i0]!r} bound {bound[i0]!r}")
    rel = np.where(bound > 0, err / np.where(bound > 0, bound, 1), 0)
    return float(np.nanmax(rel)) if rel.size else 0.0


def bf16_rne(y_f32: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(y_f32, dtype=np.float32)).to(torch.bfloat16) \
        .view(torch.int16).numpy().view(np.uint16)


def untile(tiled: np.ndarray, rows: int, row_bytes: int) -> np.ndarray:
    """Weight tile layout -> row-major (rows, row_bytes): 16 KiB tiles of
    128 rows x 128 bytes ordered (row block, chunk); the 16-byte unit j of
    row r is stored at unit position j ^ (r % 8)."""
    kc = row_bytes // 128
    a = np.asarray(tiled, dtype=np.uint8).reshape(rows // 128, kc, 128, 8, 16)
    r = np.arange(128)[:, None]
    j = np.arange(8)[None, :]
    logical = a[:, :, r, j ^ (r % 8), :]          # [rb][kc][128][8][16]
    return logical.transpose(0, 2, 1, 3, 4).reshape(rows, row_bytes)


def untile_rows(tiled: np.ndarray, rows: int, row_bytes: int, T: int) -> np.ndarray:
    """Activation tile layout with T-row tiles -> row-major (rows, row_bytes)."""
    kc = row_bytes // 128
    a = np.asarray(tiled, dtype=np.uint8).reshape(rows // T, kc, T, 8, 16)
    r = np.arange(T)[:, None]
    j = np.arange(8)[None, :]
    logical = a[:, :, r, j ^ (r % 8), :]
    return logical.transpose(0, 2, 1, 3, 4).reshape(rows, row_bytes)


def unpanel(buf: np.ndarray, rows: int, row_bytes: int, panel_bytes: int):
    """Weight panel layout -> (row-major codes (rows rounded up to 256,
    row_bytes), the scales in the flat 128x4-tile layout or None).  Per panel
    P and 128-byte chunk kc one block of panel_bytes: two 128-row tiles
    (swizzled as in `untile`), then (MXFP4) per 128-row half the chunk's two
    512-byte scale tiles."""
    kc = row_bytes // 128
    P = -(-rows // 256)
    a = np.asarray(buf, dtype=np.uint8).reshape(P, kc, panel_bytes)
    tiles = a[:, :, :32768].reshape(P, kc, 2, 128, 8, 16)
    r = np.arange(128)[:, None]
    j = np.arange(8)[None, :]
    logical = tiles[:, :, :, r, j ^ (r % 8), :]       # [P][kc][half][128][8][16]
    codes = logical.transpose(0, 2, 3, 1, 4, 5).reshape(P * 256, row_bytes)
    sf = None
    if panel_bytes > 32768:
        s = a[:, :, 32768:].reshape(P, kc, 2, 2, 512)  # [P][kc][half][tile][512]
        sf = s.transpose(0, 2, 1, 3, 4).reshape(-1)     # [row block][scale tile][512]
    return codes, sf
