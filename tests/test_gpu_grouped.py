"""Grouped (MoE) A4W4 GEMM against the oracle ("Kimi-K3-Quark-MXFP4-AttnFP8",
"Model Overview": the experts are OCP MXFP4).  Token rows arrive grouped by
expert; each group goes through its own expert's weight.  fp32 outputs within
1e-5 * sum_k |a_k w_k| of the oracle, bf16 outputs the RNE of the fp32 ones,
every output row written exactly once (rows are poisoned with NaN first).
"""
import numpy as np
import pytest
import torch

import fp8_block_scaled_dynamic_gb300 as mx
import oracle
import synth
from gpu_util import assert_codes_equal, assert_gemm_close, bf16_rne, dev

pytestmark = pytest.mark.gpu


def setup(sizes, N, K, seed):
    d = dev()
    E = len(sizes)
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    M = int(off[-1])
    x = synth.activation(M, K, seed=seed)
    ws = [synth.weight(N, K, seed=seed + 1 + e) for e in range(E)]
    panels = torch.cat([mx.mx_quantize_weight(w.to(d), layout=mx.PANEL)[0] for w in ws])
    assert panels.numel() == E * mx.mxg_weight_bytes(mx.KIND_A4W4, N, K, mx.PANEL)
    row_off = torch.from_numpy(off).to(d)
    return x, ws, panels, row_off, off


def run(x, row_off, panels, N, out_f32):
    d = dev()
    M = x.shape[0]
    y = torch.full((M, N), float("nan"), dtype=torch.float32 if out_f32 else torch.bfloat16, device=d)
    status = torch.zeros(1, dtype=torch.int32, device=d)
    mx.mx_gemm_a4w4_grouped(x.to(d), row_off, panels, n=N, out=y, out_f32=out_f32, dev_status=status,
                            weights_static=True)
    assert mx.mxg_query_status(status) == 0
    return y.cpu()


@pytest.mark.parametrize("sizes,N,K", [([0, 37, 128, 129, 300, 1], 512, 1024), ([5], 256, 512),
                                       ([200, 0, 0, 64], 768, 2048), ([1, 1, 1, 1, 1, 1, 1, 1], 384, 768),
                                       ([128, 256, 384], 1280, 512)])
def test_grouped_matches_oracle(sizes, N, K):
    x, ws, panels, row_off, off = setup(sizes, N, K, seed=sum(sizes) + N)
    y32 = run(x, row_off, panels, N, True).numpy()
    assert not np.isnan(y32).any(), "an output row was not written"
    ac, asf = oracle.mx_quantize_rows(x)
    wq = [oracle.mx_quantize_rows(w) for w in ws]
    ref, bound = oracle.gemm_a4w4_grouped(ac, asf, [q[0] for q in wq], [q[1] for q in wq], off)
    assert_gemm_close(y32, ref, bound, f"grouped {sizes} N={N} K={K}")
    y16 = run(x, row_off, panels, N, False)
    assert_codes_equal(y16.view(torch.int16).numpy().view(np.uint16), bf16_rne(y32), "bf16 = RNE(fp32)")


def test_grouped_no_tokens_launches_nothing():
    d = dev()
    N, K, E = 256, 512, 3
    panels = torch.zeros(E * mx.mxg_weight_bytes(mx.KIND_A4W4, N, K, mx.PANEL), dtype=torch.uint8, device=d)
    x = torch.zeros(0, K, dtype=torch.bfloat16, device=d)
    y = torch.zeros(0, N, dtype=torch.bfloat16, device=d)
    row_off = torch.zeros(E + 1, dtype=torch.int32, device=d)
    ws = torch.zeros(mx.mxg_grouped_workspace_bytes(0, K, E), dtype=torch.uint8, device=d)
    mx.mx_gemm_a4w4_grouped(x, row_off, panels, n=N, out=y, ws=ws)
    torch.cuda.synchronize()


def test_grouped_moe_shape_sampled_rows():
    """A synthetic expert layer of MoE size: 16 experts of gate_up shape
    (N = 2 x 2048, K = 7168), 4096 routed token rows in seeded uneven groups
    (one empty); sampled rows of every expert against the oracle."""
    rng = np.random.default_rng(7)
    sizes = rng.multinomial(4096, rng.dirichlet(np.ones(16) * 2.0)).tolist()
    sizes[3] += sizes[5]
    sizes[5] = 0
    N, K = 4096, 7168
    x, ws, panels, row_off, off = setup(sizes, N, K, seed=900)
    y32 = run(x, row_off, panels, N, True).numpy()
    assert not np.isnan(y32).any()
    for e in range(len(sizes)):
        r0, r1 = int(off[e]), int(off[e + 1])
        if r1 == r0:
            continue
        rows = np.unique(np.concatenate([[r0, r1 - 1], rng.integers(r0, r1, 3)]))
        ac, asf = oracle.mx_quantize_rows(x[torch.from_numpy(rows)].contiguous())
        wc, wsf = oracle.mx_quantize_rows(ws[e])
        ref, bound = oracle.gemm_a4w4(ac, asf, wc, wsf)
        assert_gemm_close(y32[rows], ref, bound, f"expert {e} rows {rows.tolist()}")
