"""The benchmarked step graphs themselves, checked against the oracle.

bench.py times one step of each workload as a CUDA graph built from its
launch list: weights resident in the panel layout, activations quantized
into the token-tile layout, `weights_static` GEMMs that stream their first
weight stages before their dependency wait, and the kernels of all layers
chained by programmatic dependent launch.  Here the same graphs (built by
bench.capture_step from bench.make_workload) are replayed twice, once
with fp32 outputs and once with bf16 outputs as timed, and every output of
every layer is compared with the oracle:
  * fp32: |y - ref| <= 1e-5 * sum_k |a_k w_k| per element ("Kimi-K3 DSpark
    O-Proj-only MXFP4", "Exact quantization coverage"; "Kimi-K3-DSpark-FP8-
    PTPC", "Phase 1 FP8 PTPC Quantization");
  * bf16: equal to the round-to-nearest-even of the fp32 output;
  * the device status word stays clear, both replays agree bit for bit, and
    the traced copy of the graph (the one the bench reads kernel spans from)
    gives the same bits as the plain one.
Decode-sized workloads are compared on every row, prefill-sized ones on 64
seeded sampled rows (all output channels).
"""
import numpy as np
import pytest
import torch

import bench
import fp8_block_scaled_dynamic_gb300 as mx
import synth
from gpu_util import assert_codes_equal, assert_gemm_close, bf16_rne, dev

pytestmark = pytest.mark.gpu


def replay(wl, graph, stream, bufs=None):
    """Poison the outputs, replay once, return CPU copies of the outputs."""
    for t in wl.outputs().values():
        t.fill_(float("nan") if t.is_floating_point() else 0xFF)
    if bufs is not None:
        for b in bufs:
            b.zero_()
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        graph.replay()
    stream.synchronize()
    assert mx.mxg_query_status(wl.status, stream) == 0, "a bounded device wait ran out"
    return {k: v.detach().cpu().clone() for k, v in wl.outputs().items()}


def run_graph(key, out_f32):
    d = dev()
    stream = torch.cuda.Stream(device=d)
    wl = bench.make_workload(key, mx, synth, d, out_f32=out_f32)
    with torch.cuda.stream(stream):  # eager warm-up, as the bench does
        for _, fn in wl.launches():
            fn()
    stream.synchronize()
    graph, _ = bench.capture_step(wl, stream)
    graph_t, bufs = bench.capture_step(wl, stream, traced=True)
    a = replay(wl, graph, stream)
    b = replay(wl, graph, stream)
    c = replay(wl, graph_t, stream, bufs)
    for k in a:
        assert torch.equal(a[k].view(torch.int16) if a[k].dtype == torch.bfloat16 else a[k].view(torch.int32),
                           b[k].view(torch.int16) if b[k].dtype == torch.bfloat16 else b[k].view(torch.int32)), \
            f"{key} {k}: two replays differ"
        assert torch.equal(a[k].view(torch.int16) if a[k].dtype == torch.bfloat16 else a[k].view(torch.int32),
                           c[k].view(torch.int16) if c[k].dtype == torch.bfloat16 else c[k].view(torch.int32)), \
            f"{key} {k}: the traced graph differs from the plain one"
    # every GEMM launch stamped its CTAs' entry and exit
    spans = bench.read_spans(bufs, wl.trace_labels)
    assert len(spans) == len(wl.gemm_plans())
    assert all(sp > 0 for (_, sp, _, _, _, _) in spans)
    del graph, graph_t, wl
    torch.cuda.empty_cache()
    return a


@pytest.mark.parametrize("key", ["oproj_decode", "oproj_m8", "mlp_fp8_m64", "oproj_prefill", "mlp_fp8_m8192",
                                 "moe_grouped", "mla_fp8_m64", "mla_fp8_m8192", "draft_m64"])
def test_benched_step_graph_matches_oracle(key):
    """Every output of the benched step against the oracle's version of the
    same step.  The FP8 MLP is the chain quantize -> gate_up -> SwiGLU +
    quantize -> down: its gate_up output is a bf16 tensor in both output
    modes, and its down output is held to the chain tolerance (its input
    depends on the bf16 rounding of the gate_up output, which the GEMM
    tolerance leaves open by one step; the chain is checked bit for bit on
    exactly representable data in test_gpu_swiglu.py)."""
    y32 = run_graph(key, out_f32=True)
    y16 = run_graph(key, out_f32=False)
    M = bench.workload_rows(key)
    rows = bench.sample_rows(M, 64)
    _, refs = bench.oracle_step(key, rows)
    idx = torch.from_numpy(rows)
    for name, layer, ref, bound, rule in refs:
        tol = bench.GEMM_REL_TOL if rule == "gemm" else bench.CHAIN_REL_TOL
        g32 = y32[name][layer] if layer is not None else y32[name]
        g16 = y16[name][layer] if layer is not None else y16[name]
        what = f"{key} {name} layer {layer}"
        if g32.dtype == torch.bfloat16:  # an intermediate: bf16 in both modes, bit-identical
            assert torch.equal(g32.view(torch.int16), g16.view(torch.int16)), what
        else:
            a = g32[idx].numpy()
            assert not np.isnan(a).any(), f"{what}: output not fully written"
            assert_gemm_close(a, ref, bound, what, tol=tol)
            assert_codes_equal(g16[idx].view(torch.int16).numpy().view(np.uint16), bf16_rne(a),
                               f"{what}: bf16 = RNE(fp32)")
        ok, _ = bench.bf16_interval_check(g16[idx], ref, bound, tol)
        assert ok, f"{what}: the bench's own bf16 check fails"
