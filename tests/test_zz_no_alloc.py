"""mx_gemm_a4w4_noalloc: the A4W4 GEMM for callers that cannot allocate
device memory (for example an inference engine's custom-op interface that
hands over only input and output buffers, or a serving loop that plans all
memory up front and must not allocate on its hot path).  Its scratch is a
device array owned by the library, so the caller passes no workspace.

Checked through the C ABI against the existing entry point (mx_gemm_a4w4
with a caller workspace) and against the oracle's reference: on two calls
in a row the output must agree with both within the GEMM tolerance of the
other tests (|dy| <= 1e-5 * sum_k |a_k w_k|).  A call rejected for a bad
operand must write nothing.  This file sorts last so that a
stop-at-first-failure run has already run every other test; it needs no
state from them.
"""
import ctypes

import numpy as np
import pytest
import torch

import fp8_block_scaled_dynamic_gb300 as mx
import oracle
import synth
from gpu_util import GEMM_REL_TOL, assert_gemm_close, dev

pytestmark = pytest.mark.gpu


def noalloc_entry():
    f = mx.lib().mx_gemm_a4w4_noalloc
    vp, i = ctypes.c_void_p, ctypes.c_int
    f.argtypes = [vp, vp, vp, i, vp, vp, i, i, i, vp, i, i, i, vp]
    f.restype = i
    return f


def ptr(t):
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


@pytest.mark.parametrize("M,fused,tiled", [(64, True, 1), (8, False, 0), (300, True, 0), (300, True, 2),
                                            (64, True, 2)])
def test_noalloc_matches_workspace_entry_point_on_two_calls(M, fused, tiled):
    d = dev()
    N, K = (7168, 8192) if M <= 64 else (1024, 2048)
    x = synth.activation(M, K, seed=synth.act_seed(1, 0, 0) + M)
    w = synth.weight(N, K, seed=M + 3)
    layout = {0: mx.SF_SWIZZLED, 1: mx.TILED, 2: mx.PANEL}[tiled]
    wc, wsf = mx.mx_quantize_weight(w.to(d), layout=layout)
    xd = x.to(d)
    if fused:
        ac = asf = None
        y_ref = mx.mx_gemm_a4w4(wc, wsf, x=xd, out_f32=True, weights_tiled=tiled, n=N, k=K)
    else:
        ac, asf = mx.mx_quantize_act(xd)
        y_ref = mx.mx_gemm_a4w4(wc, wsf, a_codes=ac, a_sf=asf, out_f32=True, weights_tiled=tiled,
                                n=N, k=K)
    y_ref = y_ref.cpu().numpy()
    a_c, a_s = oracle.mx_quantize_rows(x)
    w_c, w_s = oracle.mx_quantize_rows(w)
    ref, bound = oracle.gemm_a4w4(a_c, a_s, w_c, w_s)
    assert_gemm_close(y_ref, ref, bound, "mx_gemm_a4w4 with a caller workspace")

    f = noalloc_entry()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call in range(2):
        y = torch.full((M, N), float("nan"), dtype=torch.float32, device=d)
        st = f(ptr(ac), ptr(asf), ptr(xd if fused else None), K if fused else 0, ptr(wc), ptr(wsf),
               M, N, K, ptr(y), N, mx.OUT_F32, int(tiled), stream)
        assert st == 0, mx.STATUS_NAMES.get(st, st)
        torch.cuda.synchronize()
        got = y.cpu().numpy()
        assert not np.isnan(got).any(), f"call {call}: output not fully written"
        err = np.abs(got.astype(np.float64) - y_ref.astype(np.float64))
        assert (err <= GEMM_REL_TOL * bound).all(), f"call {call}: max err/bound {float((err / np.maximum(bound, 1e-300)).max())}"
        assert_gemm_close(got, ref, bound, f"mx_gemm_a4w4_noalloc call {call} vs the oracle")


def test_noalloc_rejects_shapes_beyond_its_scratch():
    d = dev()
    M, N, K = 128, 16384, 32768   # split-K with three partial slots per tile: ~25 MB
    need = mx.mxg_gemm_workspace_bytes(mx.KIND_A4W4, True, M, N, K)
    assert need > (16 << 20)
    x = torch.zeros(M, K, dtype=torch.bfloat16, device=d)
    wc = torch.zeros(N, K // 2, dtype=torch.uint8, device=d)
    wsf = torch.zeros(mx.mxg_sf_bytes(N, K), dtype=torch.uint8, device=d)
    y = torch.empty(M, N, dtype=torch.bfloat16, device=d)
    st = noalloc_entry()(None, None, ptr(x), K, ptr(wc), ptr(wsf), M, N, K, ptr(y), N, mx.OUT_BF16, 0,
                         ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 7  # MXG_ERR_WORKSPACE, before any launch


def test_noalloc_rejected_call_writes_nothing():
    """Bad operands are refused before anything is launched: the output
    buffer keeps its contents (the shared scratch is not touched either,
    which is what lets a refused call run beside one in flight)."""
    d = dev()
    M, N, K = 8, 256, 512
    x = torch.zeros(M, K, dtype=torch.bfloat16, device=d)
    wc = torch.zeros(N, K // 2, dtype=torch.uint8, device=d)
    y = torch.full((M, N), 7.0, dtype=torch.float32, device=d)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    f = noalloc_entry()
    st = f(None, None, ptr(x), K, ptr(wc), None, M, N, K, ptr(y), N, mx.OUT_F32, 0, stream)  # w_sf missing
    assert st == 1  # MXG_ERR_INVALID_ARG
    st = f(None, None, ptr(x), K, ptr(wc), ptr(wc), M, N, K, ptr(y), N, mx.OUT_F32, 5, stream)  # bad layout
    assert st == 1
    torch.cuda.synchronize()
    assert (y == 7.0).all()
