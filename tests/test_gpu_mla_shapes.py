"""FP8 PTPC at the shapes of the MLA up-projections, the other FP8 weights
of the draft layer ("Kimi-K3-DSpark-FP8-PTPC", "Phase 1 FP8 PTPC
Quantization", which lists q_b_proj and kv_b_proj among the FP8 weights).
The pages give no shapes; these are synthetic, from the usual MLA layout with
64 heads: q_b_proj 1536 -> 64 x (128 + 64) = 12288, kv_b_proj 512 -> 64 x
(128 + 128) = 16384.  Short K (512, 1536): few pipeline stages per tile, so
both dispatch variants and the split-K reduction run with small K ranges."""
import numpy as np
import pytest
import torch

import fp8_block_scaled_dynamic_gb300 as mx
import oracle
import synth
from gpu_util import assert_gemm_close, dev

pytestmark = pytest.mark.gpu

Q_B = (12288, 1536)
KV_B = (16384, 512)


@pytest.mark.parametrize("N,K", [Q_B, KV_B])
@pytest.mark.parametrize("M", [8, 64, 300, 2048])
def test_ptpc_mla_up_projection_shapes(M, N, K):
    d = dev()
    x = synth.activation(M, K, seed=M + K)
    w = synth.weight(N, K, seed=N + 11)
    qa, sa = mx.fp8_quantize_act(x.to(d))
    qw, sw = mx.fp8_quantize_weight(w.to(d), layout=mx.PANEL)
    y = mx.fp8_gemm_ptpc(qa, sa, qw, sw, out_f32=True, weights_tiled=mx.W_PANEL, k=K,
                         weights_static=True).cpu().numpy()
    rows = np.unique(np.concatenate([[0, M - 1], np.random.default_rng(M).choice(M, min(M, 24), replace=False)]))
    q_a, s_a = oracle.fp8_quantize_rows(x)
    q_w, s_w = oracle.fp8_quantize_rows(w)
    ref, bound = oracle.gemm_ptpc(q_a, s_a, q_w, s_w, rows=rows)
    assert_gemm_close(y[rows], ref, bound, f"ptpc mla {M}x{N}x{K}")


@pytest.mark.parametrize("N,K", [Q_B, KV_B])
def test_ptpc_mla_variants_agree_with_oracle_and_bf16_is_rne(N, K):
    """Both variants forced at M = 64, against the oracle on every row."""
    d = dev()
    M = 64
    x = synth.activation(M, K, seed=K + 5)
    w = synth.weight(N, K, seed=N + 13)
    qa, sa = mx.fp8_quantize_act(x.to(d))
    qw, sw = mx.fp8_quantize_weight(w.to(d))
    q_a, s_a = oracle.fp8_quantize_rows(x)
    q_w, s_w = oracle.fp8_quantize_rows(w)
    ref, bound = oracle.gemm_ptpc(q_a, s_a, q_w, s_w)
    for variant in ("full", "splitk"):
        y32 = mx.fp8_gemm_ptpc(qa, sa, qw, sw, out_f32=True, variant=variant)
        assert_gemm_close(y32.cpu().numpy(), ref, bound, f"ptpc mla {variant} {N}x{K}")
        y16 = mx.fp8_gemm_ptpc(qa, sa, qw, sw, variant=variant)
        assert torch.equal(y16.view(torch.int16), y32.to(torch.bfloat16).view(torch.int16))
