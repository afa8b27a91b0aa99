"""Split-K over CTA pairs (MXG_REDUCE_PAIR): two CTAs of a 2-CTA cluster take
the two halves of a tile's K range and the second pushes its fp32 partial
into the first one's shared memory, which adds it and writes y.  The split
points equal those of the stream-K split over 2 x tiles CTAs, so the output
must be bit-identical to the reduce-kernel path launched on that many CTAs,
and within the GEMM tolerance of the oracle."""
import numpy as np
import pytest
import torch

import fp8_block_scaled_dynamic_gb300 as mx
import oracle
import synth
from gpu_util import assert_gemm_close, dev

pytestmark = pytest.mark.gpu


def sm_count():
    return torch.cuda.get_device_properties(dev()).multi_processor_count


@pytest.mark.parametrize("M,N,K", [(8, 1024, 2048), (64, 7168, 8192), (37, 2048, 1024),
                                   (200, 1536, 1024), (1, 256, 1024)])
@pytest.mark.parametrize("layout", ["rowmajor", "panel"])
def test_a4w4_pair_bit_identical_to_reduce_kernel(M, N, K, layout):
    d = dev()
    plan = mx.mxg_plan_gemm(mx.KIND_A4W4, M, N, K, sm_count(), variant="splitk", splitk_reduce="pair")
    assert plan["pair"] == 1 and plan["ctas"] == 2 * plan["tiles"] and plan["seg_max"] == 2
    assert plan["ws_bytes"] == 0
    x = synth.activation(M, K, seed=M + N)
    w = synth.weight(N, K, seed=K + 3)
    if layout == "panel":
        wc, wsf = mx.mx_quantize_weight(w.to(d), layout=mx.PANEL)
        wt = mx.W_PANEL
    else:
        wc, wsf = mx.mx_quantize_weight(w.to(d))
        wt = mx.W_ROWMAJOR
    ac, asf = mx.mx_quantize_act(x.to(d))
    kw = dict(a_codes=ac, a_sf=asf, out_f32=True, variant="splitk", weights_tiled=wt, n=N, k=K)
    y_pair = mx.mx_gemm_a4w4(wc, wsf, splitk_reduce="pair", **kw).cpu().numpy()
    y_kern = mx.mx_gemm_a4w4(wc, wsf, splitk_reduce="kernel", ctas=plan["ctas"], **kw).cpu().numpy()
    assert (y_pair.view(np.uint32) == y_kern.view(np.uint32)).all()
    # the fused entry (bf16 x quantized inside the call) takes the same path
    y_fused = mx.mx_gemm_a4w4(wc, wsf, x=x.to(d), out_f32=True, variant="splitk", weights_tiled=wt,
                              n=N, k=K, splitk_reduce="pair").cpu().numpy()
    assert (y_fused.view(np.uint32) == y_pair.view(np.uint32)).all()
    a_c, a_s = oracle.mx_quantize_rows(x)
    w_c, w_s = oracle.mx_quantize_rows(w)
    ref, bound = oracle.gemm_a4w4(a_c, a_s, w_c, w_s)
    assert_gemm_close(y_pair, ref, bound, f"a4w4 pair {M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K", [(64, 7168, 18432), (8, 1024, 7168), (129, 2048, 1024)])
def test_ptpc_pair_bit_identical_to_reduce_kernel(M, N, K):
    d = dev()
    plan = mx.mxg_plan_gemm(mx.KIND_PTPC, M, N, K, sm_count(), variant="splitk", splitk_reduce="pair")
    assert plan["pair"] == 1
    x = synth.activation(M, K, seed=M + 5)
    w = synth.weight(N, K, seed=N + 6)
    qa, sa = mx.fp8_quantize_act(x.to(d))
    qw, sw = mx.fp8_quantize_weight(w.to(d), layout=mx.PANEL)
    kw = dict(out_f32=True, variant="splitk", weights_tiled=mx.W_PANEL, k=K)
    y_pair = mx.fp8_gemm_ptpc(qa, sa, qw, sw, splitk_reduce="pair", **kw).cpu().numpy()
    y_kern = mx.fp8_gemm_ptpc(qa, sa, qw, sw, splitk_reduce="kernel", ctas=plan["ctas"], **kw).cpu().numpy()
    assert (y_pair.view(np.uint32) == y_kern.view(np.uint32)).all()
    q_a, s_a = oracle.fp8_quantize_rows(x)
    q_w, s_w = oracle.fp8_quantize_rows(w)
    ref, bound = oracle.gemm_ptpc(q_a, s_a, q_w, s_w)
    assert_gemm_close(y_pair, ref, bound, f"ptpc pair {M}x{N}x{K}")


def test_pair_falls_back_when_tiles_exceed_half_the_sms():
    """gate_up at M = 64 has 288 tiles: no room for pairs, the reduce kernel runs."""
    d = dev()
    M, N, K = 64, 36864, 1024
    plan = mx.mxg_plan_gemm(mx.KIND_PTPC, M, N, K, sm_count(), variant="splitk", splitk_reduce="pair")
    assert plan["pair"] == 0
    x = synth.activation(M, K, seed=9)
    w = synth.weight(N, K, seed=10)
    qa, sa = mx.fp8_quantize_act(x.to(d))
    qw, sw = mx.fp8_quantize_weight(w.to(d))
    y0 = mx.fp8_gemm_ptpc(qa, sa, qw, sw, out_f32=True, variant="splitk", splitk_reduce="pair").cpu().numpy()
    y1 = mx.fp8_gemm_ptpc(qa, sa, qw, sw, out_f32=True, variant="splitk", splitk_reduce="kernel").cpu().numpy()
    assert (y0.view(np.uint32) == y1.view(np.uint32)).all()


def test_pair_bf16_output_is_rne_of_fp32():
    d = dev()
    M, N, K = 64, 7168, 8192
    x = synth.activation(M, K, seed=synth.act_seed(1, 2, 0)).to(d)
    w = synth.weight(N, K, seed=synth.SEEDS_CFG1_W[2]).to(d)
    wp, _ = mx.mx_quantize_weight(w, layout=mx.PANEL)
    kw = dict(x=x, weights_tiled=mx.W_PANEL, n=N, k=K, splitk_reduce="pair")
    y32 = mx.mx_gemm_a4w4(wp, None, out_f32=True, **kw)
    y16 = mx.mx_gemm_a4w4(wp, None, **kw)
    assert torch.equal(y16.view(torch.int16), y32.to(torch.bfloat16).view(torch.int16))
