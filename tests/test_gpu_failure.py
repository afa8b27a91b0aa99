"""Failure detection without a GPU fault: the debug_stall hook makes the
epilogue wait on a barrier that nothing arrives at; the bounded wait must
give up, the kernel must record MXG_DEV_TIMEOUT in the caller's status word
and return, and the context must stay usable for the next (correct) call."""
import numpy as np
import pytest
import torch

import fp8_block_scaled_dynamic_gb300 as mx
import oracle
import synth
from gpu_util import assert_gemm_close, dev

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("kind,variant,reduce", [(0, "full", "default"), (0, "splitk", "default"),
                                                 (1, "splitk", "default"), (1, "full", "default")])
def test_stall_times_out_then_next_call_is_correct(kind, variant, reduce):
    d = dev()
    M, N, K = 16, 512, 1024
    x = synth.activation(M, K, seed=50)
    w = synth.weight(N, K, seed=51)
    status = torch.zeros(1, dtype=torch.int32, device=d)
    ws = torch.zeros(1 << 22, dtype=torch.uint8, device=d)
    ctas = 8 if variant == "splitk" else 0  # split-K: partial sums and the reduce kernel
    if kind == 0:
        wc, wsf = mx.mx_quantize_weight(w.to(d))
        run = lambda **kw: mx.mx_gemm_a4w4(wc, wsf, x=x.to(d), out_f32=True, variant=variant, ws=ws,
                                           splitk_reduce=reduce, ctas=ctas, **kw)
        ac, asf = oracle.mx_quantize_rows(x)
        wr, wsr = oracle.mx_quantize_rows(w)
        ref, bound = oracle.gemm_a4w4(ac, asf, wr, wsr)
    else:
        qw, sw = mx.fp8_quantize_act(w.to(d))
        qa, sa = mx.fp8_quantize_act(x.to(d))
        run = lambda **kw: mx.fp8_gemm_ptpc(qa, sa, qw, sw, out_f32=True, variant=variant, ws=ws,
                                            splitk_reduce=reduce, ctas=ctas, **kw)
        qar, sar = oracle.fp8_quantize_rows(x)
        qwr, swr = oracle.fp8_quantize_rows(w)
        ref, bound = oracle.gemm_ptpc(qar, sar, qwr, swr)
    run(dev_status=status, timeout_ms=20, debug_stall=1)
    assert mx.mxg_query_status(status) == 6  # MXG_ERR_TIMEOUT
    assert int(status.item()) == 0           # cleared by the query
    y = run(dev_status=status)
    assert mx.mxg_query_status(status) == 0
    assert_gemm_close(y.cpu().numpy(), ref, bound, "after timeout")


@pytest.mark.parametrize("kind", [0, 1])
def test_stall_on_cta_pairs_times_out_then_next_call_is_correct(kind):
    """The same on CTA pairs (2-SM MMAs, clusters of two): both CTAs of a
    pair give up, meet at the cluster barrier, release their TMEM together
    and return; the next call on pairs is correct."""
    d = dev()
    M, N, K = 256, 512, 1024
    x = synth.activation(M, K, seed=52)
    w = synth.weight(N, K, seed=53)
    status = torch.zeros(1, dtype=torch.int32, device=d)
    assert mx.mxg_plan_gemm(kind, M, N, K, 152, variant="full", cta_pair=True)["cta_pair"] == 1
    if kind == 0:
        wc, wsf = mx.mx_quantize_weight(w.to(d))
        run = lambda **kw: mx.mx_gemm_a4w4(wc, wsf, x=x.to(d), out_f32=True, variant="full", cta_pair=True, **kw)
        ac, asf = oracle.mx_quantize_rows(x)
        wr, wsr = oracle.mx_quantize_rows(w)
        ref, bound = oracle.gemm_a4w4(ac, asf, wr, wsr)
    else:
        qw, sw = mx.fp8_quantize_act(w.to(d))
        qa, sa = mx.fp8_quantize_act(x.to(d))
        run = lambda **kw: mx.fp8_gemm_ptpc(qa, sa, qw, sw, out_f32=True, variant="full", cta_pair=True, **kw)
        qar, sar = oracle.fp8_quantize_rows(x)
        qwr, swr = oracle.fp8_quantize_rows(w)
        ref, bound = oracle.gemm_ptpc(qar, sar, qwr, swr)
    run(dev_status=status, timeout_ms=20, debug_stall=1)
    assert mx.mxg_query_status(status) == 6  # MXG_ERR_TIMEOUT
    y = run(dev_status=status)
    assert mx.mxg_query_status(status) == 0
    assert_gemm_close(y.cpu().numpy(), ref, bound, "after timeout, pairs")


def test_stall_in_fused_quantizer_times_out_then_next_call_is_correct():
    """debug_stall = 2: the activation quantizer of a fused call with more
    than 512 token rows (rows streamed through shared memory) waits on a
    barrier that nothing arrives at.  Every CTA gives up, lets its copies in
    flight land, records MXG_DEV_TIMEOUT and leaves NaN scales (E8M0 0xFF)
    on its rows, so every output row is NaN; the next call is correct."""
    d = dev()
    M, N, K = 600, 512, 1024
    x = synth.activation(M, K, seed=54)
    w = synth.weight(N, K, seed=55)
    status = torch.zeros(1, dtype=torch.int32, device=d)
    wc, wsf = mx.mx_quantize_weight(w.to(d))
    run = lambda **kw: mx.mx_gemm_a4w4(wc, wsf, x=x.to(d), out_f32=True, **kw)
    y = run(dev_status=status, timeout_ms=20, debug_stall=2)
    assert mx.mxg_query_status(status) == 6  # MXG_ERR_TIMEOUT
    assert np.isnan(y.cpu().numpy()).all()
    y = run(dev_status=status)
    assert mx.mxg_query_status(status) == 0
    ac, asf = oracle.mx_quantize_rows(x)
    wr, wsr = oracle.mx_quantize_rows(w)
    ref, bound = oracle.gemm_a4w4(ac, asf, wr, wsr)
    assert_gemm_close(y.cpu().numpy(), ref, bound, "after a quantizer timeout")
