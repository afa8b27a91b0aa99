"""GPU parity of the step between the packed gate_up projection and the down
projection: swiglu_fp8_quantize (SwiGLU of a [gate | up] row fused with the
per-token FP8 quantization of h = bf16(silu(gate) * up)), against the
oracle ("Kimi-K3-DSpark-FP8-PTPC", "Phase 1 FP8 PTPC Quantization": gate_proj
and up_proj packed into one gate_up_proj; dynamic per-token FP8 activations).

The oracle and the kernel form silu in binary32 one IEEE operation at a time
with the same published exp method, so h, the codes and the scales are
compared bit for bit -- on every bf16 gate value, on random rows in the
row-major and token-tile layouts, and on special rows.  Then the whole FP8
MLP chain of the bench (quantize, gate_up, this step, down; one CUDA graph)
runs on exactly representable data, where the gate_up output is exact on
both sides, so that every intermediate of the chain is checked bit for bit
and the down output within the GEMM tolerance.
"""
import numpy as np
import pytest
import torch

import bench
import fp8_block_scaled_dynamic_gb300 as mx
import oracle
import synth
from gpu_util import assert_codes_equal, assert_gemm_close, bf16_rne, dev, untile_rows

pytestmark = pytest.mark.gpu


def bits16(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def assert_bf16_equal(got, want, what):
    """bf16 bit patterns equal, any NaN matching any NaN."""
    gn = (got & 0x7FFF) > 0x7F80
    wn = (want & 0x7FFF) > 0x7F80
    assert (gn == wn).all(), f"{what}: NaN positions differ"
    assert_codes_equal(np.where(gn, 0, got), np.where(wn, 0, want), what)


def run_and_check(gu, T=0):
    d = dev()
    M, I = gu.shape[0], gu.shape[1] // 2
    h = torch.empty(M, I, dtype=torch.bfloat16, device=d)
    q, s = mx.swiglu_fp8_quantize(gu.to(d), T, h=h)
    h_ref, q_ref, s_ref = oracle.swiglu_fp8_quantize_rows(gu)
    assert_bf16_equal(bits16(h), h_ref, "h")
    qc = q.cpu().numpy()
    if T:
        rows = -(-M // T) * T
        qc = untile_rows(qc, rows, I, T)[:M]
    assert_codes_equal(qc, q_ref, f"codes (tile rows {T})")
    sc = s.cpu().numpy()
    assert (np.isnan(sc) == np.isnan(s_ref)).all()
    assert_codes_equal(np.where(np.isnan(sc), 0, sc).view(np.uint32),
                       np.where(np.isnan(s_ref), 0, s_ref).view(np.uint32), "scales")


@pytest.mark.parametrize("up", ["one", "random"])
def test_every_bf16_gate_value(up):
    """All 65536 bf16 patterns as gate (16 rows of 4096), with up = 1 (h =
    bf16(silu(g))) or random: h, codes and scales bit-exact; the two rows
    holding infinities and NaNs get NaN scales and zero codes."""
    gate = torch.arange(65536, dtype=torch.int32).to(torch.int16).view(torch.bfloat16).reshape(16, 4096)
    if up == "one":
        u = torch.ones(16, 4096, dtype=torch.bfloat16)
    else:
        u = synth.bf16_randn(16, 4096, seed=3, sigma=2.0)
    run_and_check(torch.cat([gate, u], dim=1))


@pytest.mark.parametrize("M,I", [(1, 128), (7, 2048), (64, 18432), (300, 1024), (129, 384)])
@pytest.mark.parametrize("T", [0, 16, 64, 128, 256])
def test_random_rows(M, I, T):
    gu = synth.bf16_randn(M, 2 * I, seed=M * 7 + I + T, sigma=4.0, outlier_frac=0.001)
    run_and_check(gu, T)


@pytest.mark.parametrize("I", [86016, 90112, 102400])
def test_wide_rows(I):
    """Rows at the widest I that keeps the 32 KiB silu table beside the row
    in shared memory (86016), and wider ones formed without it, up to the
    largest I the call takes: the same bits either way."""
    gu = synth.bf16_randn(2, 2 * I, seed=I, sigma=4.0, outlier_frac=0.001)
    run_and_check(gu)
    run_and_check(gu, 16)


def test_special_rows():
    """A zero row (s = 1, codes +-0), a row whose gates all saturate to -0
    (h = -0 everywhere), rows with an infinite or NaN up value, a row with
    huge gates (silu(g) = g) and one with subnormal inputs."""
    I = 256
    rows = []
    rows.append(torch.zeros(2 * I))
    rows.append(torch.cat([torch.full((I,), -500.0), torch.full((I,), 3.0)]))
    r = torch.randn(2 * I)
    r[I + 5] = float("inf")
    rows.append(r)
    r = torch.randn(2 * I)
    r[I + 77] = float("nan")
    rows.append(r)
    rows.append(torch.cat([torch.full((I,), 3.0e38), torch.linspace(-1, 1, I)]))
    rows.append(torch.full((2 * I,), 1e-39))
    gu = torch.stack(rows).to(torch.bfloat16)
    run_and_check(gu)
    run_and_check(gu, 16)


# ---------------------------------------------------------------- the chain
def exact_mlp_inputs(M, H, I, seed):
    """x (M, H) and W_gu (2I, H) with integer values whose gate_up products
    are exact in binary32 and bf16: every row of x and of W_gu holds one 448
    (so every per-token and per-channel FP8 scale is exactly 1) in columns
    where the other operand is zero; elsewhere x has 32 values in {+-1, +-2}
    and W_gu values in [-3, 3], so |gate_up| <= 192."""
    rng = np.random.default_rng(seed)
    x = np.zeros((M, H), np.float32)
    x[np.arange(M), np.arange(M) % 64] = 448.0
    for m in range(M):
        cols = rng.choice(np.arange(2048, H), 32, replace=False)
        x[m, cols] = rng.choice(np.array([-2.0, -1.0, 1.0, 2.0], np.float32), 32)
    w = np.zeros((2 * I, H), np.int8)
    w[:, 2048:] = rng.integers(-3, 4, (2 * I, H - 2048), dtype=np.int8)
    wt = torch.from_numpy(w).to(torch.bfloat16)
    wt[torch.arange(2 * I), 64 + torch.arange(2 * I) % 1024] = 448.0
    return torch.from_numpy(x).to(torch.bfloat16), wt


def test_mlp_chain_graph_bit_exact_on_exact_data():
    """The bench's FP8 MLP chain graph (bench.MlpFp8, bench.capture_step) on
    exactly representable inputs: the gate_up output equals the oracle's
    exactly, the SwiGLU step's codes and scales (in the down GEMM's token
    tiles) equal the oracle's bit for bit, and the down output is within
    1e-5 * sum|a w| of the oracle's, its bf16 twin the RNE of the fp32."""
    d = dev()
    M, H, I = 64, 7168, synth.MLP_I
    x, w_gu = exact_mlp_inputs(M, H, I, seed=1)
    w_down = synth.weight(H, I, seed=synth.SEED_CFG3_DOWN)
    outs = {}
    for out_f32 in (True, False):
        stream = torch.cuda.Stream(device=d)
        wl = bench.MlpFp8(mx, synth, d, M, name="exact", out_f32=out_f32, x=x, w_gu=w_gu, w_down=w_down)
        with torch.cuda.stream(stream):
            for _, fn in wl.launches():
                fn()
        stream.synchronize()
        graph, _ = bench.capture_step(wl, stream)
        for t in wl.outputs().values():
            t.zero_()
        with torch.cuda.stream(stream):
            graph.replay()
        stream.synchronize()
        assert mx.mxg_query_status(wl.status, stream) == 0
        outs[out_f32] = {k: v.detach().cpu().clone() for k, v in wl.outputs().items()}
        Td = wl.Td
        del graph, wl
        torch.cuda.empty_cache()
    qa, sa = oracle.fp8_quantize_rows(x)
    qg, sg = oracle.fp8_quantize_rows(w_gu)
    assert (sa == 1.0).all() and (sg == 1.0).all()
    ref_g, _ = oracle.gemm_ptpc(qa, sa, qg, sg)
    assert (ref_g == np.round(ref_g)).all() and np.abs(ref_g).max() <= 256
    g16 = torch.from_numpy(ref_g.astype(np.float32)).to(torch.bfloat16)
    for o in outs.values():
        assert_codes_equal(bits16(o["yg"]), bits16(g16), "gate_up output")
    _, qh, sh = oracle.swiglu_fp8_quantize_rows(g16)
    q_gpu = untile_rows(outs[True]["qh"].numpy(), -(-M // Td) * Td, I, Td)[:M]
    assert_codes_equal(q_gpu, qh, "SwiGLU codes in the down GEMM's token tiles")
    assert_codes_equal(outs[True]["sh"].numpy().view(np.uint32), sh.view(np.uint32), "SwiGLU scales")
    qd, sd = oracle.fp8_quantize_rows(w_down)
    ref_d, bound_d = oracle.gemm_ptpc(qh, sh, qd, sd)
    y32 = outs[True]["yd"].numpy()
    assert_gemm_close(y32, ref_d, bound_d, "down output of the chain")
    assert_codes_equal(bits16(outs[False]["yd"]), bf16_rne(y32), "bf16 = RNE(fp32)")
