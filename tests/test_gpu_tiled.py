"""The weight tile layout (16 KiB tiles of 128 rows x 128 bytes, pre-swizzled,
fetched by the GEMM with one bulk copy per stage): the quantizers must emit
exactly the oracle's codes re-arranged, and GEMMs on tiled weights must give
bit-identical outputs to the same GEMMs on row-major weights."""
import numpy as np
import pytest
import torch

import fp8_block_scaled_dynamic_gb300 as mx
import oracle
import synth
from gpu_util import assert_codes_equal, assert_gemm_close, dev, np_u8, untile, untile_rows

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("N,K", [(128, 256), (384, 1024), (7168, 8192)])
def test_mx_weight_tiled_codes(N, K):
    w = synth.weight(N, K, seed=N + K)
    codes, sf = mx.mx_quantize_weight(w.to(dev()), layout=mx.TILED)
    c_ref, s_ref = oracle.mx_quantize_rows(w)
    assert_codes_equal(untile(np_u8(codes).reshape(-1), N, K // 2), c_ref, "tiled codes")
    assert_codes_equal(np_u8(sf), oracle.sf_swizzle(s_ref), "tiled scales")


@pytest.mark.parametrize("N,K", [(128, 128), (256, 7168), (384, 18432)])
def test_fp8_weight_tiled_and_rowmajor(N, K):
    w = synth.weight(N, K, seed=N * 3 + K)
    q_ref, s_ref = oracle.fp8_quantize_rows(w)
    q, s = mx.fp8_quantize_weight(w.to(dev()), layout=mx.SF_ROWMAJOR)
    assert_codes_equal(np_u8(q), q_ref, "fp8 row-major weight")
    assert (s.cpu().numpy().view(np.uint32) == s_ref.view(np.uint32)).all()
    qt, st = mx.fp8_quantize_weight(w.to(dev()), layout=mx.TILED)
    assert_codes_equal(untile(np_u8(qt).reshape(-1), N, K), q_ref, "fp8 tiled weight")
    assert (st.cpu().numpy().view(np.uint32) == s_ref.view(np.uint32)).all()


def test_tiled_layout_rejects_bad_shapes():
    d = dev()
    w = synth.weight(200, 256, seed=1).to(d)
    with pytest.raises(mx.MxgError):
        mx.mx_quantize_weight(w, layout=mx.TILED)           # N % 128
    w = synth.weight(128, 384, seed=1).to(d)
    with pytest.raises(mx.MxgError):
        mx.mx_quantize_weight(w, layout=mx.TILED)           # K % 256 for MXFP4


@pytest.mark.parametrize("M,N,K", [(8, 384, 1024), (64, 1024, 2048), (300, 512, 768), (1, 256, 512)])
@pytest.mark.parametrize("variant", ["full", "splitk"])
def test_a4w4_tiled_weights_bit_identical(M, N, K, variant):
    if K % 256:
        pytest.skip("MXFP4 tiles need K % 256 == 0")
    d = dev()
    x = synth.activation(M, K, seed=M + 7)
    w = synth.weight(N, K, seed=N + 9)
    wc, wsf = mx.mx_quantize_weight(w.to(d))
    wt, wtsf = mx.mx_quantize_weight(w.to(d), layout=mx.TILED)
    y0 = mx.mx_gemm_a4w4(wc, wsf, x=x.to(d), out_f32=True, variant=variant).cpu().numpy()
    y1 = mx.mx_gemm_a4w4(wt, wtsf, x=x.to(d), out_f32=True, variant=variant,
                         weights_tiled=True).cpu().numpy()
    assert (y0.view(np.uint32) == y1.view(np.uint32)).all()
    ac, asf = oracle.mx_quantize_rows(x)
    wr, wsr = oracle.mx_quantize_rows(w)
    ref, bound = oracle.gemm_a4w4(ac, asf, wr, wsr)
    assert_gemm_close(y1, ref, bound, f"tiled a4w4 {variant}")


@pytest.mark.parametrize("M,N,K", [(8, 384, 1024), (64, 1024, 2048), (300, 512, 768)])
@pytest.mark.parametrize("variant", ["full", "splitk"])
def test_ptpc_tiled_weights_bit_identical(M, N, K, variant):
    d = dev()
    x = synth.activation(M, K, seed=M + 17)
    w = synth.weight(N, K, seed=N + 19)
    qa, sa = mx.fp8_quantize_act(x.to(d))
    qw, sw = mx.fp8_quantize_weight(w.to(d))
    qt, st = mx.fp8_quantize_weight(w.to(d), layout=mx.TILED)
    y0 = mx.fp8_gemm_ptpc(qa, sa, qw, sw, out_f32=True, variant=variant).cpu().numpy()
    y1 = mx.fp8_gemm_ptpc(qa, sa, qt, st, out_f32=True, variant=variant, weights_tiled=True).cpu().numpy()
    assert (y0.view(np.uint32) == y1.view(np.uint32)).all()


def test_a4w4_decode_m64_tiled_full_size():
    d = dev()
    x = synth.activation(64, synth.OPROJ_K, seed=synth.act_seed(1, 1, 0))
    w = synth.weight(synth.OPROJ_N, synth.OPROJ_K, seed=synth.SEEDS_CFG1_W[1])
    wt, wtsf = mx.mx_quantize_weight(w.to(d), layout=mx.TILED)
    y = mx.mx_gemm_a4w4(wt, wtsf, x=x.to(d), out_f32=True, weights_tiled=True).cpu().numpy()
    ac, asf = oracle.mx_quantize_rows(x)
    wr, wsr = oracle.mx_quantize_rows(w)
    ref, bound = oracle.gemm_a4w4(ac, asf, wr, wsr)
    assert_gemm_close(y, ref, bound, "cfg1 layer 1, tiled weights")


# ------------------------------------------------------------------ activation tiles
@pytest.mark.parametrize("M,T", [(8, 16), (64, 64), (37, 64), (300, 128), (129, 256)])
def test_act_tiled_codes(M, T):
    d = dev()
    K = 1024
    x = synth.activation(M, K, seed=M * 11 + T)
    codes, sf = mx.mx_quantize_act_tiled(x.to(d), T)
    c_ref, s_ref = oracle.mx_quantize_rows(x)
    rows_pad = -(-M // T) * T
    got = untile_rows(np_u8(codes), rows_pad, K // 2, T)[:M]
    assert_codes_equal(got, c_ref, "tiled act codes")
    assert_codes_equal(np_u8(sf), oracle.sf_swizzle(s_ref), "tiled act scales")
    q, s = mx.fp8_quantize_act_tiled(x.to(d), T)
    q_ref, s8_ref = oracle.fp8_quantize_rows(x)
    assert_codes_equal(untile_rows(np_u8(q), rows_pad, K, T)[:M], q_ref, "tiled fp8 act")
    assert (s.cpu().numpy().view(np.uint32) == s8_ref.view(np.uint32)).all()


@pytest.mark.parametrize("kind", ["a4w4", "ptpc"])
@pytest.mark.parametrize("M,variant", [(8, "splitk"), (64, "splitk"), (200, "splitk"), (300, "full"), (64, "full")])
def test_gemm_on_tiled_activations_bit_identical(kind, M, variant):
    d = dev()
    N, K = 512, 1024
    x = synth.activation(M, K, seed=M + 31).to(d)
    w = synth.weight(N, K, seed=N + 33).to(d)
    sm = torch.cuda.get_device_properties(d).multi_processor_count
    plan = mx.mxg_plan_gemm(mx.KIND_A4W4 if kind == "a4w4" else mx.KIND_PTPC, M, N, K, sm, variant=variant)
    T = plan["bn"] if plan["variant"] == 2 else 128
    if kind == "a4w4":
        wt, wtsf = mx.mx_quantize_weight(w, layout=mx.TILED)
        ac, asf = mx.mx_quantize_act(x)
        act, asft = mx.mx_quantize_act_tiled(x, T)
        y0 = mx.mx_gemm_a4w4(wt, wtsf, a_codes=ac, a_sf=asf, out_f32=True, variant=variant, weights_tiled=True)
        y1 = mx.mx_gemm_a4w4(wt, wtsf, a_codes=act, a_sf=asft, out_f32=True, variant=variant,
                             weights_tiled=True, act_tile_rows=T, m=M)
    else:
        qt, st = mx.fp8_quantize_weight(w, layout=mx.TILED)
        qa, sa = mx.fp8_quantize_act(x)
        qat, sat = mx.fp8_quantize_act_tiled(x, T)
        y0 = mx.fp8_gemm_ptpc(qa, sa, qt, st, out_f32=True, variant=variant, weights_tiled=True)
        y1 = mx.fp8_gemm_ptpc(qat, sat, qt, st, out_f32=True, variant=variant, weights_tiled=True,
                              act_tile_rows=T)
    assert (y0.cpu().numpy().view(np.uint32) == y1.cpu().numpy().view(np.uint32)).all()


def test_act_tile_rows_must_match_plan():
    d = dev()
    x = synth.activation(64, 1024, seed=5).to(d)
    w = synth.weight(512, 1024, seed=6).to(d)
    wt, wtsf = mx.mx_quantize_weight(w, layout=mx.TILED)
    act, asft = mx.mx_quantize_act_tiled(x, 32)   # the split-K plan for M=64 uses 64-row tiles
    with pytest.raises(mx.MxgError):
        mx.mx_gemm_a4w4(wt, wtsf, a_codes=act, a_sf=asft, weights_tiled=True, act_tile_rows=32, m=64)
