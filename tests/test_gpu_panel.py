"""The weight panel layout (256-row panels, each 128-byte chunk holding the
codes of both 128-row halves and, for MXFP4, their scales, so that a
full-tile GEMM stage fetches its whole weight operand with one bulk copy):
the quantizers must emit exactly the oracle's codes and scales re-arranged,
with zero codes in the padding rows, and GEMMs on panel weights must give
outputs bit-identical to the same GEMMs on row-major or tiled weights, in
both dispatch variants."""
import numpy as np
import pytest
import torch

import fp8_block_scaled_dynamic_gb300 as mx
import oracle
import synth
from gpu_util import assert_codes_equal, assert_gemm_close, dev, np_u8, unpanel

pytestmark = pytest.mark.gpu

MX_PANEL_BYTES, F8_PANEL_BYTES = 34816, 32768


@pytest.mark.parametrize("N,K", [(128, 256), (384, 1024), (640, 2048), (7168, 8192)])
def test_mx_weight_panel_codes_and_scales(N, K):
    w = synth.weight(N, K, seed=N * 5 + K)
    codes, sf = mx.mx_quantize_weight(w.to(dev()), layout=mx.PANEL)
    assert sf is None
    assert codes.numel() == mx.mxg_weight_bytes(mx.KIND_A4W4, N, K, mx.PANEL) \
        == -(-N // 256) * (K // 256) * MX_PANEL_BYTES
    c_ref, s_ref = oracle.mx_quantize_rows(w)
    got_c, got_sf = unpanel(np_u8(codes), N, K // 2, MX_PANEL_BYTES)
    assert_codes_equal(got_c[:N], c_ref, "panel codes")
    assert not got_c[N:].any(), "padding rows must hold zero codes"
    want_sf = oracle.sf_swizzle(s_ref)
    assert_codes_equal(got_sf[:want_sf.size], want_sf, "panel scales")


@pytest.mark.parametrize("N,K", [(128, 128), (384, 1024), (256, 7168)])
def test_fp8_weight_panel_bytes(N, K):
    w = synth.weight(N, K, seed=N * 7 + K)
    q, s = mx.fp8_quantize_weight(w.to(dev()), layout=mx.PANEL)
    assert q.numel() == mx.mxg_weight_bytes(mx.KIND_PTPC, N, K, mx.PANEL) == -(-N // 256) * (K // 128) * F8_PANEL_BYTES
    q_ref, s_ref = oracle.fp8_quantize_rows(w)
    got, _ = unpanel(np_u8(q), N, K, F8_PANEL_BYTES)
    assert_codes_equal(got[:N], q_ref, "fp8 panel bytes")
    assert not got[N:].any(), "padding rows must hold zero bytes"
    assert (s.cpu().numpy().view(np.uint32) == s_ref.view(np.uint32)).all()


def test_panel_layout_rejects_bad_shapes():
    d = dev()
    w = synth.weight(128, 384, seed=2).to(d)
    with pytest.raises(ValueError):
        mx.mx_quantize_weight(w, layout=mx.PANEL)          # K % 256 for MXFP4
    assert mx.mxg_weight_bytes(mx.KIND_A4W4, 128, 384, mx.PANEL) == 0


@pytest.mark.parametrize("M,N,K", [(8, 384, 1024), (64, 1024, 2048), (300, 512, 768),
                                   (300, 384, 1024), (1, 256, 512), (520, 640, 2048)])
@pytest.mark.parametrize("variant", ["full", "splitk"])
def test_a4w4_panel_weights_bit_identical(M, N, K, variant):
    if K % 256:
        pytest.skip("MXFP4 panels need K % 256 == 0")
    d = dev()
    x = synth.activation(M, K, seed=M + 71)
    w = synth.weight(N, K, seed=N + 73)
    wc, wsf = mx.mx_quantize_weight(w.to(d))
    wp, _ = mx.mx_quantize_weight(w.to(d), layout=mx.PANEL)
    y0 = mx.mx_gemm_a4w4(wc, wsf, x=x.to(d), out_f32=True, variant=variant).cpu().numpy()
    y1 = mx.mx_gemm_a4w4(wp, None, x=x.to(d), out_f32=True, variant=variant,
                         weights_tiled=mx.W_PANEL, n=N, k=K).cpu().numpy()
    assert (y0.view(np.uint32) == y1.view(np.uint32)).all()
    ac, asf = oracle.mx_quantize_rows(x)
    wr, wsr = oracle.mx_quantize_rows(w)
    ref, bound = oracle.gemm_a4w4(ac, asf, wr, wsr)
    assert_gemm_close(y1, ref, bound, f"panel a4w4 {variant}")


@pytest.mark.parametrize("M,N,K", [(8, 384, 1024), (64, 1024, 2048), (300, 512, 768), (300, 384, 1152)])
@pytest.mark.parametrize("variant", ["full", "splitk"])
def test_ptpc_panel_weights_bit_identical(M, N, K, variant):
    d = dev()
    x = synth.activation(M, K, seed=M + 77)
    w = synth.weight(N, K, seed=N + 79)
    qa, sa = mx.fp8_quantize_act(x.to(d))
    qw, sw = mx.fp8_quantize_weight(w.to(d))
    qp, sp = mx.fp8_quantize_weight(w.to(d), layout=mx.PANEL)
    y0 = mx.fp8_gemm_ptpc(qa, sa, qw, sw, out_f32=True, variant=variant).cpu().numpy()
    y1 = mx.fp8_gemm_ptpc(qa, sa, qp, sp, out_f32=True, variant=variant, weights_tiled=mx.W_PANEL,
                          k=K).cpu().numpy()
    assert (y0.view(np.uint32) == y1.view(np.uint32)).all()


@pytest.mark.parametrize("ctas", [0, 3])
def test_a4w4_panel_splitk_fused(ctas):
    """The split-K path takes one 128-row half of a panel as its weight tile;
    on the fused path (x quantized inside the call) panels and weight tiles
    give the same bits."""
    d = dev()
    M, N, K = 64, 1536, 4096
    x = synth.activation(M, K, seed=91).to(d)
    w = synth.weight(N, K, seed=92).to(d)
    wt, wtsf = mx.mx_quantize_weight(w, layout=mx.TILED)
    wp, _ = mx.mx_quantize_weight(w, layout=mx.PANEL)
    y0 = mx.mx_gemm_a4w4(wt, wtsf, x=x, out_f32=True, weights_tiled=mx.W_TILED, variant="splitk", ctas=ctas)
    y1 = mx.mx_gemm_a4w4(wp, None, x=x, out_f32=True, weights_tiled=mx.W_PANEL, n=N, k=K, variant="splitk",
                         ctas=ctas)
    assert (y0.cpu().numpy().view(np.uint32) == y1.cpu().numpy().view(np.uint32)).all()


@pytest.mark.parametrize("kind", ["a4w4", "ptpc"])
def test_prefill_full_size_panels_match_tiles(kind):
    """The prefill workload (M = 8192 tokens, o_proj 7168 x 8192): the output
    on panel weights equals the output on 128-row weight tiles bit for bit,
    and sampled rows match the oracle."""
    d = dev()
    M, N, K = 8192, synth.OPROJ_N, synth.OPROJ_K
    x = synth.activation(M, K, seed=synth.act_seed(1, 0, 0) + 5)
    w = synth.weight(N, K, seed=synth.SEEDS_CFG1_W[0])
    xd, wd = x.to(d), w.to(d)
    if kind == "a4w4":
        wt, wtsf = mx.mx_quantize_weight(wd, layout=mx.TILED)
        wp, _ = mx.mx_quantize_weight(wd, layout=mx.PANEL)
        ac, asf = mx.mx_quantize_act_tiled(xd, 128)
        y0 = mx.mx_gemm_a4w4(wt, wtsf, a_codes=ac, a_sf=asf, weights_tiled=mx.W_TILED,
                             act_tile_rows=128, m=M, out_f32=True)
        y1 = mx.mx_gemm_a4w4(wp, None, a_codes=ac, a_sf=asf, weights_tiled=mx.W_PANEL,
                             act_tile_rows=128, m=M, n=N, k=K, out_f32=True)
    else:
        qt, st = mx.fp8_quantize_weight(wd, layout=mx.TILED)
        qp, sp = mx.fp8_quantize_weight(wd, layout=mx.PANEL)
        qa, sa = mx.fp8_quantize_act_tiled(xd, 128)
        y0 = mx.fp8_gemm_ptpc(qa, sa, qt, st, weights_tiled=mx.W_TILED, act_tile_rows=128, out_f32=True)
        y1 = mx.fp8_gemm_ptpc(qa, sa, qp, sp, weights_tiled=mx.W_PANEL, act_tile_rows=128, k=K,
                              out_f32=True)
    torch.cuda.synchronize()
    assert torch.equal(y0.view(torch.int32), y1.view(torch.int32))
    rows = np.sort(np.random.default_rng(11).choice(M, 24, replace=False))
    rows[0], rows[-1] = 0, M - 1
    y = y1[torch.from_numpy(rows).to(d)].cpu().numpy()
    if kind == "a4w4":
        ac_r, as_r = oracle.mx_quantize_rows(x)
        wc_r, ws_r = oracle.mx_quantize_rows(w)
        ref, bound = oracle.gemm_a4w4(ac_r, as_r, wc_r, ws_r, rows=rows)
    else:
        qa_r, sa_r = oracle.fp8_quantize_rows(x)
        qw_r, sw_r = oracle.fp8_quantize_rows(w)
        ref, bound = oracle.gemm_ptpc(qa_r, sa_r, qw_r, sw_r, rows=rows)
    assert_gemm_close(y, ref, bound, f"prefill {kind} on panels, sampled rows")
