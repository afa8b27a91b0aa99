"""CPU-side checks of the C ABI: the library loads without a GPU, exports
every function include/mxgemm.h declares, rejects bad arguments before any
launch, and its dispatcher (pure host logic) plans the stream-K split the
way an independent simulation says it must."""
import ctypes
import os
import re

import numpy as np
import pytest

import fp8_block_scaled_dynamic_gb300 as mx

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    src = ""
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            src += open(os.path.join(ROOT, "include", f)).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z_0-9]*\s*\*?\s*([a-z_][a-z_0-9]*)\s*\(",
                       src, flags=re.M)
    return sorted(set(names))


def test_library_exports_every_declared_symbol():
    names = declared_functions()
    assert {"mx_quantize_weight", "mx_quantize_act", "mx_gemm_a4w4", "fp8_quantize_act",
            "fp8_gemm_ptpc"} <= set(names)
    L = mx.lib()
    for n in names:
        assert hasattr(L, n), f"{n} declared in include/ but not exported"


def test_sf_bytes():
    assert mx.mxg_sf_bytes(7168, 8192, mx.SF_ROWMAJOR) == 7168 * 256
    assert mx.mxg_sf_bytes(7168, 8192, mx.SF_SWIZZLED) == 7168 * 256
    assert mx.mxg_sf_bytes(8, 8192, mx.SF_SWIZZLED) == 128 * 256
    assert mx.mxg_sf_bytes(129, 256, mx.SF_SWIZZLED) == 256 * 8
    assert mx.mxg_sf_bytes(0, 256, mx.SF_SWIZZLED) == 0
    assert mx.mxg_sf_bytes(7168, 8192, mx.TILED) == 7168 * 256
    assert mx.mxg_sf_bytes(7168, 8192, mx.PANEL) == 0      # the scales sit inside the panels


def test_weight_bytes():
    # row-major and tile layouts: N x row bytes
    assert mx.mxg_weight_bytes(mx.KIND_A4W4, 7168, 8192, mx.SF_SWIZZLED) == 7168 * 4096
    assert mx.mxg_weight_bytes(mx.KIND_PTPC, 7168, 8192, mx.TILED) == 7168 * 8192
    # panels: ceil(N / 256) panels x (row bytes / 128) chunks x (32 KiB codes + 2 KiB MXFP4 scales)
    assert mx.mxg_weight_bytes(mx.KIND_A4W4, 7168, 8192, mx.PANEL) == 28 * 32 * 34816
    assert mx.mxg_weight_bytes(mx.KIND_A4W4, 384, 1024, mx.PANEL) == 2 * 4 * 34816
    assert mx.mxg_weight_bytes(mx.KIND_PTPC, 384, 1152, mx.PANEL) == 2 * 9 * 32768
    # the codes plus the swizzled scales, re-arranged: the same bytes when N % 256 == 0
    assert mx.mxg_weight_bytes(mx.KIND_A4W4, 7168, 8192, mx.PANEL) == \
        7168 * 4096 + mx.mxg_sf_bytes(7168, 8192, mx.SF_SWIZZLED)
    assert mx.mxg_weight_bytes(mx.KIND_A4W4, 128, 384, mx.PANEL) == 0   # MXFP4 panels need K % 256
    assert mx.mxg_weight_bytes(2, 128, 256, mx.PANEL) == 0


def test_status_strings():
    L = mx.lib()
    for code, name in mx.STATUS_NAMES.items():
        assert L.mxg_status_string(code).decode() == name


FAKE = 1 << 20  # a 16-byte aligned pointer value; nothing is dereferenced on these paths


@pytest.mark.parametrize("args,want", [
    ((FAKE, 8, 100, 100, FAKE, FAKE, None), 2),   # K % 128
    ((None, 8, 128, 128, FAKE, FAKE, None), 1),   # null input
    ((FAKE, 0, 128, 128, FAKE, FAKE, None), 1),   # M = 0
    ((FAKE, 8, 128, 64, FAKE, FAKE, None), 1),    # ld < K
    ((FAKE + 2, 8, 128, 128, FAKE, FAKE, None), 3),  # misaligned x
    ((FAKE, 8, 128, 132, FAKE, FAKE, None), 3),   # ld*2 not a multiple of 16
    ((FAKE, 8, 128, 128, FAKE + 8, FAKE, None), 3),  # misaligned codes
])
def test_quantizer_argument_errors_before_launch(args, want):
    assert mx.lib().mx_quantize_act(*args) == want


def test_gemm_argument_errors_before_launch():
    L = mx.lib()
    o = mx.GemmOpts()
    # N % 128
    assert L.fp8_gemm_ptpc(FAKE, FAKE, FAKE, FAKE, 8, 100, 128, FAKE, 100, 0, ctypes.byref(o), None) == 2
    # bad output dtype
    assert L.fp8_gemm_ptpc(FAKE, FAKE, FAKE, FAKE, 8, 128, 128, FAKE, 128, 7, ctypes.byref(o), None) == 1
    # ldy < N
    assert L.mx_gemm_a4w4(FAKE, FAKE, None, 0, FAKE, FAKE, 8, 256, 256, FAKE, 128, 0, None, None) == 1
    # fused path without x
    assert L.mx_gemm_a4w4(None, None, None, 0, FAKE, FAKE, 8, 256, 256, FAKE, 256, 0, None, None) == 1
    # misaligned y
    assert L.mx_gemm_a4w4(FAKE, FAKE, None, 0, FAKE, FAKE, 8, 256, 256, FAKE + 4, 256, 0, None, None) == 3
    # bad variant
    o.variant = 9
    assert L.mx_gemm_a4w4(FAKE, FAKE, None, 0, FAKE, FAKE, 8, 256, 256, FAKE, 256, 0, ctypes.byref(o), None) == 1
    o.variant = 0
    # bad weight layout / split-K reduction
    o.weights_tiled = 3
    assert L.mx_gemm_a4w4(FAKE, FAKE, None, 0, FAKE, FAKE, 8, 256, 256, FAKE, 256, 0, ctypes.byref(o), None) == 1
    o.weights_tiled = 0
    o.splitk_reduce = 5
    assert L.fp8_gemm_ptpc(FAKE, FAKE, FAKE, FAKE, 8, 128, 128, FAKE, 128, 0, ctypes.byref(o), None) == 1
    o.splitk_reduce = 0
    # w_sf may be NULL only for weight panels
    assert L.mx_gemm_a4w4(FAKE, FAKE, None, 0, FAKE, None, 8, 256, 256, FAKE, 256, 0, ctypes.byref(o), None) == 1


def test_weight_quantizer_layout_errors_before_launch():
    L = mx.lib()
    L.mx_quantize_weight.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                     ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p]
    # unknown layout
    assert L.mx_quantize_weight(FAKE, 128, 256, 256, FAKE, FAKE, 4, None) == 1
    # MXFP4 panels and tiles need K % 256 == 0; tiles also N % 128 == 0
    assert L.mx_quantize_weight(FAKE, 128, 384, 384, FAKE, None, mx.PANEL, None) == 2
    assert L.mx_quantize_weight(FAKE, 128, 384, 384, FAKE, FAKE, mx.TILED, None) == 2
    assert L.mx_quantize_weight(FAKE, 200, 256, 256, FAKE, FAKE, mx.TILED, None) == 2
    # scales are required except in panels, whose scales sit inside them
    assert L.mx_quantize_weight(FAKE, 128, 256, 256, FAKE, None, mx.SF_SWIZZLED, None) == 1
    # FP8 weights: no MXFP4 row-major-scales-only layout
    assert L.fp8_quantize_weight(FAKE, 128, 256, 256, FAKE, FAKE, mx.SF_SWIZZLED, None) == 1
    assert L.fp8_quantize_weight(FAKE, 200, 256, 256, FAKE, FAKE, mx.TILED, None) == 2


def owner_sim(U, G):
    """Independent statement of the even stream-K cut: CTA c takes units
    [floor(c U / G), floor((c+1) U / G))."""
    own = np.empty(U, np.int64)
    for c in range(G):
        own[(c * U) // G:((c + 1) * U) // G] = c
    return own


@pytest.mark.parametrize("kind,M,N,K,sm", [(0, 8, 7168, 8192, 152), (0, 64, 7168, 8192, 152),
                                           (1, 64, 36864, 7168, 152), (1, 64, 7168, 18432, 152),
                                           (0, 200, 1024, 2048, 7), (1, 1, 128, 128, 152),
                                           (1, 64, 16384, 512, 152), (1, 64, 12288, 1536, 152),
                                           (0, 64, 12288, 1536, 152), (1, 8, 4096, 2048, 152)])
def test_plan_splitk_matches_simulation(kind, M, N, K, sm):
    """The stream-K cut over min(SMs, units) CTAs -- or, when the tiles fit
    in one wave and their K takes no more stages than a stream-K CTA's share
    plus the 7 stages a chained reduce kernel costs, one CTA per whole tile
    (no partial sums)."""
    p = mx.mxg_plan_gemm(kind, M, N, K, sm, variant="splitk")
    assert p["variant"] == 2 and p["bm"] == 128
    assert p["bn"] >= M and p["bn"] in (16, 32, 64, 128, 256) and (p["bn"] // 2 < M or p["bn"] == 16)
    kcol = 256 if kind == 0 else 128  # K values in one 128-byte column
    KB = -(-(-(-K // kcol)) // 2)      # split-K stages take two columns
    assert p["kblocks"] == KB
    tiles = (N // 128) * (-(-M // p["bn"]))
    assert p["tiles"] == tiles
    U = tiles * KB
    G = min(sm, U)
    own = owner_sim(U, G)
    seg = max(len(set(own[t * KB:(t + 1) * KB])) for t in range(tiles))
    if tiles <= sm and seg > 1 and KB <= -(-U // G) + 7:
        G, seg = tiles, 1
        own = owner_sim(U, G)
        assert max(len(set(own[t * KB:(t + 1) * KB])) for t in range(tiles)) == 1
    assert p["ctas"] == G
    assert p["seg_max"] == seg
    if seg > 1:
        assert p["ws_bytes"] >= tiles * seg * p["bn"] * 128 * 4


def test_plan_full_tile_for_large_m():
    p = mx.mxg_plan_gemm(0, 8192, 7168, 8192, 152)
    assert p["variant"] == 1 and p["bn"] == 256 and p["tiles"] == 64 * 28 and p["ctas"] == 152
    assert p["ws_bytes"] == 0 and p["cta_pair"] == 0
    p = mx.mxg_plan_gemm(1, 300, 384, 1024, 152, variant="splitk")
    assert p["variant"] == 2 and p["bn"] == 256 and p["tiles"] == 3 * 2


def test_plan_errors():
    with pytest.raises(mx.MxgError):
        mx.mxg_plan_gemm(0, 8, 7168, 8000, 152)  # K % 128
    with pytest.raises(mx.MxgError):
        mx.mxg_plan_gemm(2, 8, 7168, 8192, 152)  # kind


def test_only_the_reduce_kernel_is_a_split_k_reduction():
    """The split-K partials are summed by the reduce kernel; other values of
    splitk_reduce are refused before anything is launched."""
    L = mx.lib()
    o = mx.GemmOpts()
    for v in (2, 3, 4, -1):
        o.splitk_reduce = v
        assert L.fp8_gemm_ptpc(FAKE, FAKE, FAKE, FAKE, 8, 128, 128, FAKE, 128, 0, ctypes.byref(o), None) == 1
    p = mx.mxg_plan_gemm(0, 64, 7168, 8192, 152, variant="splitk")
    assert p["cta_pair"] == 0 and p["ws_bytes"] == p["tiles"] * p["seg_max"] * p["bn"] * 128 * 4


@pytest.mark.parametrize("kind,M,N,K,want", [
    # o_proj (A4W4, 28 full tiles per 128 tokens): split-K up to M = 128, full tile beyond
    (0, 8, 7168, 8192, 2), (0, 64, 7168, 8192, 2), (0, 128, 7168, 8192, 2),
    (0, 192, 7168, 8192, 1), (0, 512, 7168, 8192, 1), (0, 8192, 7168, 8192, 1),
    # FP8 gate_up (144 full tiles >= 0.9 x 152 SMs at any M): full tile
    (1, 8, 36864, 7168, 1), (1, 64, 36864, 7168, 1), (1, 8192, 36864, 7168, 1),
    # FP8 down (long K): split-K up to M = 256, full tile beyond
    (1, 64, 7168, 18432, 2), (1, 256, 7168, 18432, 2), (1, 320, 7168, 18432, 1),
])
def test_dispatcher_rule(kind, M, N, K, want):
    """The automatic variant follows the GB300 measurements of quantizer + GEMM:
    a full wave of 128 x 256 tiles -> full tile; otherwise split-K for M <= 128,
    and up to M = 256 when K exceeds 64 128-byte columns."""
    assert mx.mxg_plan_gemm(kind, M, N, K, 152)["variant"] == want


@pytest.mark.parametrize("args,want", [
    ((FAKE, 8, 100, 200, 0, FAKE, FAKE, None, 0), 2),      # I % 128
    ((FAKE, 8, 204800, 409600, 0, FAKE, FAKE, None, 0), 2),  # h of a row beyond shared memory
    ((None, 8, 128, 256, 0, FAKE, FAKE, None, 0), 1),       # null input
    ((FAKE, 0, 128, 256, 0, FAKE, FAKE, None, 0), 1),       # M = 0
    ((FAKE, 8, 128, 200, 0, FAKE, FAKE, None, 0), 1),       # ldgu < 2I
    ((FAKE, 8, 128, 256, 48, FAKE, FAKE, None, 0), 1),      # tile height not a power of two in 16..256
    ((FAKE, 8, 128, 256, 0, FAKE, FAKE, FAKE, 64), 1),      # ldh < I
    ((FAKE + 2, 8, 128, 256, 0, FAKE, FAKE, None, 0), 3),   # misaligned gate_up
    ((FAKE, 8, 128, 260, 0, FAKE, FAKE, None, 0), 3),       # ldgu * 2 not a multiple of 16
    ((FAKE, 8, 128, 256, 0, FAKE, FAKE + 4, None, 0), 3),   # misaligned scale
])
def test_swiglu_argument_errors_before_launch(args, want):
    assert mx.lib().swiglu_fp8_quantize(*args, None) == want


def test_grouped_argument_errors_before_launch():
    L = mx.lib()
    o = mx.GemmOpts()
    f = L.mx_gemm_a4w4_grouped
    # x, ldx, row_off, E, w, M, N, K, y, ldy, dtype, opts, stream
    assert f(None, 512, FAKE, 4, FAKE, 64, 256, 512, FAKE, 256, 0, ctypes.byref(o), None) == 1  # no x
    assert f(FAKE, 512, FAKE, 0, FAKE, 64, 256, 512, FAKE, 256, 0, ctypes.byref(o), None) == 1  # E = 0
    assert f(FAKE, 256, FAKE, 4, FAKE, 64, 256, 512, FAKE, 256, 0, ctypes.byref(o), None) == 1  # ldx < K
    assert f(FAKE, 384, FAKE, 4, FAKE, 64, 256, 384, FAKE, 256, 0, ctypes.byref(o), None) == 2  # K % 256
    assert f(FAKE, 512, FAKE, 4, FAKE, 64, 200, 512, FAKE, 256, 0, ctypes.byref(o), None) == 2  # N % 128
    assert f(FAKE, 512, FAKE, 4, FAKE, 64, 256, 512, FAKE, 256, 0, ctypes.byref(o), None) == 7  # no workspace
    assert f(FAKE, 512, FAKE, 4, FAKE, 64, 256, 512, FAKE, 256, 0, None, None) == 7
    o.variant = 2  # split-K is not a grouped variant
    assert f(FAKE, 512, FAKE, 4, FAKE, 64, 256, 512, FAKE, 256, 0, ctypes.byref(o), None) == 1
    # workspace: token tiles for ceil(M / 128) + E tiles, plus the tile offsets
    assert mx.mxg_grouped_workspace_bytes(300, 1024, 4) >= (3 + 4) * 128 * (1024 // 2 + 1024 // 32)
    assert mx.mxg_grouped_workspace_bytes(300, 1024, 0) == 0


@pytest.mark.parametrize("kind,M,N,K,pair,tiles,ctas", [
    # one token tile: one CTA per 128 x 256 tile even when pairs are asked for
    (1, 64, 36864, 7168, 0, 144, 144), (0, 100, 7168, 8192, 0, 28, 28),
    # two token tiles or more: CTA pairs over 256 x 256 tiles, one pair per two SMs
    (0, 192, 7168, 8192, 1, 28, 56), (0, 8192, 7168, 8192, 1, 32 * 28, 152),
    (1, 8192, 36864, 7168, 1, 32 * 144, 152), (1, 300, 7168, 18432, 1, 2 * 28, 112),
])
def test_full_tile_cta_pairs(kind, M, N, K, pair, tiles, ctas):
    """On request (cta_pair) the full tile runs on CTA pairs (2-SM MMAs,
    256-token x 256-channel tiles) when there are two token tiles or more;
    the grid is even and holds at most one pair per two SMs.  Without the
    request it never does."""
    p = mx.mxg_plan_gemm(kind, M, N, K, 152, variant="full", cta_pair=True)
    assert p["variant"] == 1 and p["cta_pair"] == pair and p["tiles"] == tiles and p["ctas"] == ctas
    assert p["bm"] == (256 if pair else 128) and p["bn"] == 256
    if pair:
        assert p["ctas"] % 2 == 0
    q = mx.mxg_plan_gemm(kind, M, N, K, 152, variant="full")
    assert q["cta_pair"] == 0 and q["bm"] == 128


def test_cta_pair_argument_checked():
    """cta_pair must be 0 or 1, and 0 for the grouped GEMM; refused before launch."""
    L = mx.lib()
    o = mx.GemmOpts(cta_pair=2)
    assert L.fp8_gemm_ptpc(FAKE, FAKE, FAKE, FAKE, 8, 128, 128, FAKE, 128, 0, ctypes.byref(o), None) == 1
