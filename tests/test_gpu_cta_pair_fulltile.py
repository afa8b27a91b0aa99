"""The full-tile GEMM on CTA pairs (mxg_gemm_opts.cta_pair): clusters of two
CTAs issuing 2-SM MMAs (tcgen05 cta_group::2) over 256-token x 256-channel
tiles, each CTA holding 128 token rows and one 128-row half of the weight
tile.  What is computed is the same GEMM ("Kimi-K3 DSpark O-Proj-only MXFP4",
"Exact quantization coverage"; "Kimi-K3-DSpark-FP8-PTPC", "Phase 1 FP8 PTPC
Quantization"): fp32 outputs within 1e-5 * sum_k |a_k w_k| of the oracle,
bf16 outputs the RNE of the fp32 ones, and -- the MMAs accumulate every
output element over K in the same order as one CTA per tile does -- bit for
bit the single-CTA result.  Cases cover an odd number of token tiles (the
last pair's second CTA has no token rows), ragged M, a last weight tile only
half filled, and every weight layout.
"""
import numpy as np
import pytest
import torch

import fp8_block_scaled_dynamic_gb300 as mx
import oracle
import synth
from gpu_util import assert_codes_equal, assert_gemm_close, bf16_rne, dev

pytestmark = pytest.mark.gpu

SHAPES = [(256, 512, 512), (384, 768, 1024), (1000, 1280, 2048), (300, 640, 768)]
LAYOUTS = [mx.W_ROWMAJOR, mx.W_TILED, mx.W_PANEL]


def a4w4(x, w, layout, pair, out_f32=True, tiles=False):
    d = dev()
    N, K = w.shape
    if layout == mx.W_PANEL:
        wc, wsf = mx.mx_quantize_weight(w.to(d), layout=mx.PANEL)[0], None
    elif layout == mx.W_TILED:
        wc, wsf = mx.mx_quantize_weight(w.to(d), layout=mx.TILED)
    else:
        wc, wsf = mx.mx_quantize_weight(w.to(d))
    kw = dict(out_f32=out_f32, variant="full", weights_tiled=layout, cta_pair=pair, n=N, k=K)
    if tiles:
        ac, asf = mx.mx_quantize_act_tiled(x.to(d), 128)
        return mx.mx_gemm_a4w4(wc, wsf, a_codes=ac, a_sf=asf, act_tile_rows=128, m=x.shape[0], **kw)
    ac, asf = mx.mx_quantize_act(x.to(d))
    return mx.mx_gemm_a4w4(wc, wsf, a_codes=ac, a_sf=asf, **kw)


def ptpc(x, w, layout, pair, out_f32=True):
    d = dev()
    N, K = w.shape
    if layout == mx.W_PANEL:
        qw, sw = mx.fp8_quantize_weight(w.to(d), layout=mx.PANEL)
    elif layout == mx.W_TILED:
        qw, sw = mx.fp8_quantize_weight(w.to(d), layout=mx.TILED)
    else:
        qw, sw = mx.fp8_quantize_act(w.to(d))
    qa, sa = mx.fp8_quantize_act(x.to(d))
    return mx.fp8_gemm_ptpc(qa, sa, qw, sw, out_f32=out_f32, variant="full", weights_tiled=layout,
                            cta_pair=pair, k=K)


def check(kind, M, N, K, layout, tiles=False):
    sm = torch.cuda.get_device_properties(dev()).multi_processor_count
    assert mx.mxg_plan_gemm(kind, M, N, K, sm, variant="full", cta_pair=True)["cta_pair"] == 1
    x = synth.activation(M, K, seed=M + 3 * N + K)
    w = synth.weight(N, K, seed=M + 3 * N + K + 1)
    if kind == mx.KIND_A4W4:
        run = lambda pair, f32=True: a4w4(x, w, layout, pair, f32, tiles)
        a, sa_ = oracle.mx_quantize_rows(x)
        b, sb = oracle.mx_quantize_rows(w)
        ref, bound = oracle.gemm_a4w4(a, sa_, b, sb)
    else:
        run = lambda pair, f32=True: ptpc(x, w, layout, pair, f32)
        a, sa_ = oracle.fp8_quantize_rows(x)
        b, sb = oracle.fp8_quantize_rows(w)
        ref, bound = oracle.gemm_ptpc(a, sa_, b, sb)
    y_pair = run(True).cpu().numpy()
    what = f"kind {kind} {M}x{N}x{K} layout {layout} tiles {tiles}"
    assert_gemm_close(y_pair, ref, bound, what)
    y_one = run(False).cpu().numpy()
    assert_codes_equal(y_pair.view(np.uint32), y_one.view(np.uint32), what + ": pair = one CTA per tile")
    y16 = run(True, False)
    assert_codes_equal(y16.view(torch.int16).cpu().numpy().view(np.uint16), bf16_rne(y_pair), what + ": bf16")


@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("layout", LAYOUTS)
def test_a4w4_pairs(M, N, K, layout):
    check(mx.KIND_A4W4, M, N, K, layout)


@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("layout", LAYOUTS)
def test_ptpc_pairs(M, N, K, layout):
    check(mx.KIND_PTPC, M, N, K, layout)


@pytest.mark.parametrize("M", [384, 1000])
def test_a4w4_pairs_token_tiles(M):
    """Activations in 128-row token tiles with weight panels (the bench's layout)."""
    check(mx.KIND_A4W4, M, 768, 1024, mx.W_PANEL, tiles=True)


def test_a4w4_pairs_fused_activations():
    """bf16 activations quantized inside the call, then the pair kernel."""
    d = dev()
    M, N, K = 520, 512, 1024
    x = synth.activation(M, K, seed=5)
    w = synth.weight(N, K, seed=6)
    wc, wsf = mx.mx_quantize_weight(w.to(d))
    y = mx.mx_gemm_a4w4(wc, wsf, x=x.to(d), out_f32=True, variant="full", cta_pair=True).cpu().numpy()
    a, sa_ = oracle.mx_quantize_rows(x)
    b, sb = oracle.mx_quantize_rows(w)
    ref, bound = oracle.gemm_a4w4(a, sa_, b, sb)
    assert_gemm_close(y, ref, bound, "fused A4W4 on CTA pairs")


def test_pairs_prefill_shape_sampled_rows():
    """o_proj at a prefill size (M = 2048, N = 7168, K = 8192; 8 x 28 pair
    tiles over 76 pairs, several tiles per pair), panels and token tiles;
    sampled rows against the oracle, all rows against the single-CTA run."""
    d = dev()
    M, N, K = 2048, 7168, 8192
    x = synth.activation(M, K, seed=11, row_scale=True)
    w = synth.weight(N, K, seed=12)
    wc = mx.mx_quantize_weight(w.to(d), layout=mx.PANEL)[0]
    ac, asf = mx.mx_quantize_act_tiled(x.to(d), 128)
    kw = dict(a_codes=ac, a_sf=asf, act_tile_rows=128, m=M, n=N, k=K, out_f32=True, variant="full",
              weights_tiled=mx.W_PANEL, weights_static=True)
    y_pair = mx.mx_gemm_a4w4(wc, None, cta_pair=True, **kw).cpu().numpy()
    y_one = mx.mx_gemm_a4w4(wc, None, cta_pair=False, **kw).cpu().numpy()
    assert_codes_equal(y_pair.view(np.uint32), y_one.view(np.uint32), "pair = one CTA per tile")
    rng = np.random.default_rng(3)
    rows = np.unique(np.concatenate([[0, 127, 128, 255, 256, M - 1], rng.integers(0, M, 10)]))
    a, sa_ = oracle.mx_quantize_rows(x[torch.from_numpy(rows)].contiguous())
    b, sb = oracle.mx_quantize_rows(w)
    ref, bound = oracle.gemm_a4w4(a, sa_, b, sb)
    assert_gemm_close(y_pair[rows], ref, bound, "pairs, sampled rows")
