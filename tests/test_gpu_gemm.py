"""GPU GEMMs vs the CPU oracle: |y_f32 - ref| <= 1e-5 * sum_k |a_k w_k| per
element, and the bf16 output equal to the bf16 rounding of the fp32 output.

A4W4: "Kimi-K3 DSpark O-Proj-only MXFP4", "Exact quantization coverage"
(dynamic MXFP4 activations with A4W4 dispatch on the (7168, 8192) o_proj).
PTPC: "Kimi-K3-DSpark-FP8-PTPC", "Phase 1 FP8 PTPC Quantization" (E4M3
weights with per-output-channel scales, dynamic per-token activations;
gate_proj and up_proj packed into one gate_up GEMM).
"""
import numpy as np
import pytest
import torch

import fp8_block_scaled_dynamic_gb300 as mx
import oracle
import synth
from gpu_util import assert_codes_equal, assert_gemm_close, bf16_rne, dev, np_u8

pytestmark = pytest.mark.gpu


def pack_codes(c):
    return (c[:, 0::2] | (c[:, 1::2] << 4)).astype(np.uint8)


def to_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev())


# ------------------------------------------------------------------ one-hot
@pytest.mark.parametrize("variant", ["full", "splitk"])
def test_a4w4_one_hot_pins_nibble_order_and_scale_layout(variant):
    """A single nonzero code at (m, k) in A and (n, k) in W must light only
    y[m][n], with the value v(a) v(w) 2^(ea+ew-254).  Positions cover both
    nibbles, several 32-groups and 128-groups, and all four 32-row quarters
    of a 128-row scale tile."""
    M, N, K = 160, 384, 512
    G = K // 32
    cases = [(0, 0, 0), (1, 1, 1), (33, 130, 37), (70, 255, 100), (100, 383, 511),
             (127, 64, 260), (128, 200, 383), (159, 97, 222)]
    rng = np.random.default_rng(3)
    for (m, n, k) in cases:
        a = np.zeros((M, K), np.uint8)
        w = np.zeros((N, K), np.uint8)
        a[m, k] = 0x5   # 3.0
        w[n, k] = 0xE   # -4.0
        a_sf = rng.integers(110, 140, (M, G)).astype(np.uint8)
        w_sf = rng.integers(110, 140, (N, G)).astype(np.uint8)
        y = mx.mx_gemm_a4w4(to_dev(pack_codes(w)), to_dev(oracle.sf_swizzle(w_sf)),
                            a_codes=to_dev(pack_codes(a)), a_sf=to_dev(oracle.sf_swizzle(a_sf)),
                            out_f32=True, variant=variant).cpu().numpy()
        want = np.zeros((M, N))
        want[m, n] = 3.0 * -4.0 * 2.0 ** (int(a_sf[m, k // 32]) + int(w_sf[n, k // 32]) - 254)
        nz = np.argwhere(y != 0)
        assert nz.tolist() == [[m, n]], (m, n, k, nz[:5].tolist())
        assert y[m, n] == want[m, n], (m, n, k, y[m, n], want[m, n])


@pytest.mark.parametrize("variant", ["full", "splitk"])
def test_ptpc_one_hot(variant):
    M, N, K = 140, 256, 384
    for (m, n, k) in [(0, 0, 0), (5, 129, 31), (77, 255, 200), (139, 17, 383)]:
        qa = np.zeros((M, K), np.uint8)
        qw = np.zeros((N, K), np.uint8)
        qa[m, k] = 0x44   # 3.0 in E4M3 (exp 8 -> 2^1 * 1.5)
        qw[n, k] = 0xB8   # -1.0
        sa = np.linspace(0.5, 2.0, M).astype(np.float32)
        sw = np.linspace(0.25, 4.0, N).astype(np.float32)
        y = mx.fp8_gemm_ptpc(to_dev(qa), to_dev(sa), to_dev(qw), to_dev(sw), out_f32=True,
                             variant=variant).cpu().numpy()
        nz = np.argwhere(y != 0)
        assert nz.tolist() == [[m, n]], (m, n, k, nz[:5].tolist())
        want = np.float32(np.float32(np.float32(3.0 * -1.0) * sa[m]) * sw[n])
        assert y[m, n] == want, (y[m, n], want)


# ------------------------------------------------------------------ A4W4 parity
def quant_pair(M, N, K, seed, row_scale=False):
    x = synth.activation(M, K, seed=seed, row_scale=row_scale)
    w = synth.weight(N, K, seed=seed + 1)
    return x, w


def run_a4w4(x, w, variant, fused=True, out_f32=True, ctas=0):
    d = dev()
    wc, wsf = mx.mx_quantize_weight(w.to(d))
    if fused:
        return mx.mx_gemm_a4w4(wc, wsf, x=x.to(d), out_f32=out_f32, variant=variant, ctas=ctas)
    ac, asf = mx.mx_quantize_act(x.to(d))
    return mx.mx_gemm_a4w4(wc, wsf, a_codes=ac, a_sf=asf, out_f32=out_f32, variant=variant, ctas=ctas)


def oracle_a4w4(x, w, rows=None):
    ac, asf = oracle.mx_quantize_rows(x)
    wc, wsf = oracle.mx_quantize_rows(w)
    return oracle.gemm_a4w4(ac, asf, wc, wsf, rows=rows)


@pytest.mark.parametrize("M,N,K", [(1, 128, 256), (8, 384, 1024), (37, 256, 384),
                                   (64, 1024, 2048), (129, 512, 768), (300, 640, 1280)])
@pytest.mark.parametrize("variant", ["full", "splitk"])
def test_a4w4_small_shapes(M, N, K, variant):
    x, w = quant_pair(M, N, K, seed=M + N + K)
    y32 = run_a4w4(x, w, variant).cpu().numpy()
    ref, bound = oracle_a4w4(x, w)
    assert_gemm_close(y32, ref, bound, f"a4w4 {variant} {M}x{N}x{K}")
    y16 = run_a4w4(x, w, variant, out_f32=False)
    assert_codes_equal(y16.view(torch.int16).cpu().numpy().view(np.uint16), bf16_rne(y32),
                       "bf16 output = RNE(fp32 output)")


@pytest.mark.parametrize("ctas", [1, 3, 7, 57, 152, 500])
def test_a4w4_splitk_cta_counts(ctas):
    x, w = quant_pair(24, 768, 2048, seed=9)
    y = run_a4w4(x, w, "splitk", ctas=ctas).cpu().numpy()
    ref, bound = oracle_a4w4(x, w)
    assert_gemm_close(y, ref, bound, f"splitk ctas={ctas}")


def test_a4w4_fused_equals_prequantized_and_is_deterministic():
    x, w = quant_pair(64, 1024, 4096, seed=77)
    a = run_a4w4(x, w, "splitk", fused=True).cpu().numpy()
    b = run_a4w4(x, w, "splitk", fused=False).cpu().numpy()
    c = run_a4w4(x, w, "splitk", fused=True).cpu().numpy()
    assert (a.view(np.uint32) == b.view(np.uint32)).all()
    assert (a.view(np.uint32) == c.view(np.uint32)).all()


@pytest.mark.parametrize("M,N,K,ctas", [(64, 1024, 4096, 0), (8, 7168, 8192, 0), (37, 768, 2048, 7),
                                         (200, 512, 2048, 0), (256, 1280, 1024, 57), (24, 640, 640, 0),
                                         (64, 2048, 4096, 1), (16, 3072, 2048, 5)])
def test_a4w4_splitk_fused_equals_prequantized_and_repeats(M, N, K, ctas):
    """The split-K partial tiles are summed in slot order by the reduce
    kernel, so the bits do not depend on timing: the fused path (x given,
    quantized inside the call) equals the pre-quantized one, and a second
    call equals the first.  With few CTAs every CTA walks many tiles (items),
    so the epilogue feeds the next item's scales while it stores the one
    before (two TMEM accumulators)."""
    d = dev()
    x, w = quant_pair(M, N, K, seed=M * 7 + N)
    wc, wsf = mx.mx_quantize_weight(w.to(d))
    ac, asf = mx.mx_quantize_act(x.to(d))
    outs = {"pre": mx.mx_gemm_a4w4(wc, wsf, a_codes=ac, a_sf=asf, out_f32=True, variant="splitk", ctas=ctas),
            "fused": mx.mx_gemm_a4w4(wc, wsf, x=x.to(d), out_f32=True, variant="splitk", ctas=ctas),
            "again": mx.mx_gemm_a4w4(wc, wsf, a_codes=ac, a_sf=asf, out_f32=True, variant="splitk", ctas=ctas)}
    ref, bound = oracle_a4w4(x, w)
    y0 = outs["pre"].cpu().numpy()
    assert_gemm_close(y0, ref, bound, f"splitk {M}x{N}x{K} ctas={ctas}")
    for m, y in outs.items():
        assert (y.cpu().numpy().view(np.uint32) == y0.view(np.uint32)).all(), m


@pytest.mark.parametrize("M,N,K,ctas", [(64, 1024, 2048, 0), (5, 7168, 1024, 0), (130, 384, 896, 0),
                                         (64, 2048, 2048, 1), (24, 1536, 4096, 5)])
def test_ptpc_splitk_matches_oracle_and_repeats(M, N, K, ctas):
    d = dev()
    x, w = quant_pair(M, N, K, seed=M + 3 * N)
    qw, sw = mx.fp8_quantize_act(w.to(d))
    qa, sa = mx.fp8_quantize_act(x.to(d))
    y0 = mx.fp8_gemm_ptpc(qa, sa, qw, sw, out_f32=True, variant="splitk", ctas=ctas).cpu().numpy()
    y1 = mx.fp8_gemm_ptpc(qa, sa, qw, sw, out_f32=True, variant="splitk", ctas=ctas).cpu().numpy()
    assert (y0.view(np.uint32) == y1.view(np.uint32)).all()
    ref, bound = oracle_ptpc(x, w)
    assert_gemm_close(y0, ref, bound, f"ptpc splitk {M}x{N}x{K} ctas={ctas}")


def test_a4w4_decode_m8_full_size():
    # single o_proj layer, M = 8 (1 verified + 7 drafted tokens), N = 7168, K = 8192
    x = synth.activation(8, synth.OPROJ_K, seed=synth.act_seed(0, 0, 0))
    w = synth.weight(synth.OPROJ_N, synth.OPROJ_K, seed=synth.SEED_CFG0_W)
    y = run_a4w4(x, w, "auto").cpu().numpy()
    ref, bound = oracle_a4w4(x, w)
    assert_gemm_close(y, ref, bound, "cfg0 M=8")


@pytest.mark.parametrize("layer", [0, 4])
def test_a4w4_decode_m64_layers(layer):
    x = synth.activation(64, synth.OPROJ_K, seed=synth.act_seed(1, layer, 0))
    w = synth.weight(synth.OPROJ_N, synth.OPROJ_K, seed=synth.SEEDS_CFG1_W[layer])
    y = run_a4w4(x, w, "auto").cpu().numpy()
    ref, bound = oracle_a4w4(x, w)
    assert_gemm_close(y, ref, bound, f"cfg1 layer {layer}")


def test_a4w4_prefill_m8192_sampled_rows():
    x = synth.activation(8192, synth.OPROJ_K, seed=synth.act_seed(2, 0, 0), row_scale=True)
    w = synth.weight(synth.OPROJ_N, synth.OPROJ_K, seed=synth.SEED_CFG2_W)
    y = run_a4w4(x, w, "auto").cpu().numpy()
    rows = np.sort(np.random.default_rng(2).choice(8192, 48, replace=False))
    rows[0], rows[-1] = 0, 8191
    ref, bound = oracle_a4w4(x, w, rows=rows)
    assert_gemm_close(y[rows], ref, bound, "cfg2 sampled rows")


# ------------------------------------------------------------------ PTPC parity
def run_ptpc(x, w, variant, out_f32=True, ctas=0):
    d = dev()
    qw, sw = mx.fp8_quantize_act(w.to(d))
    qa, sa = mx.fp8_quantize_act(x.to(d))
    return mx.fp8_gemm_ptpc(qa, sa, qw, sw, out_f32=out_f32, variant=variant, ctas=ctas)


def oracle_ptpc(x, w, rows=None):
    qa, sa = oracle.fp8_quantize_rows(x)
    qw, sw = oracle.fp8_quantize_rows(w)
    return oracle.gemm_ptpc(qa, sa, qw, sw, rows=rows)


@pytest.mark.parametrize("M,N,K", [(1, 128, 128), (8, 384, 1024), (37, 256, 384),
                                   (64, 1024, 2048), (129, 512, 768), (300, 640, 1280)])
@pytest.mark.parametrize("variant", ["full", "splitk"])
def test_ptpc_small_shapes(M, N, K, variant):
    x, w = quant_pair(M, N, K, seed=3 * M + N + K)
    y32 = run_ptpc(x, w, variant).cpu().numpy()
    ref, bound = oracle_ptpc(x, w)
    assert_gemm_close(y32, ref, bound, f"ptpc {variant} {M}x{N}x{K}")
    y16 = run_ptpc(x, w, variant, out_f32=False)
    assert_codes_equal(y16.view(torch.int16).cpu().numpy().view(np.uint16), bf16_rne(y32),
                       "bf16 output = RNE(fp32 output)")


@pytest.mark.parametrize("M", [64, 8192])
def test_ptpc_mlp_pair_sampled_rows(M):
    # gate_up: K = 7168 -> N = 2 x 18432; down: K = 18432 -> N = 7168
    rng = np.random.default_rng(M)
    rows = np.sort(rng.choice(M, min(M, 12), replace=False))
    xg = synth.activation(M, 7168, seed=synth.act_seed(3, 0, 0))
    wg = synth.weight(2 * synth.MLP_I, 7168, seed=synth.SEED_CFG3_GATE_UP)
    y = run_ptpc(xg, wg, "auto").cpu().numpy()
    ref, bound = oracle_ptpc(xg, wg, rows=rows)
    assert_gemm_close(y[rows], ref, bound, f"gate_up M={M}")
    xd = synth.activation(M, synth.MLP_I, seed=synth.act_seed(3, 0, 1))
    wd = synth.weight(7168, synth.MLP_I, seed=synth.SEED_CFG3_DOWN)
    y = run_ptpc(xd, wd, "auto").cpu().numpy()
    ref, bound = oracle_ptpc(xd, wd, rows=rows)
    assert_gemm_close(y[rows], ref, bound, f"down M={M}")


@pytest.mark.parametrize("kind,lo,hi", [(0, 1000.0, 20000.0), (1, 500.0, 10000.0)])
def test_mma_loop_peak_is_plausible(kind, lo, hi):
    """The measurement utility runs and lands between a tenth of and above the
    nominal dense rate (13.5 PF/s E2M1, 4.5 PF/s E4M3 on GB300)."""
    t = mx.mxg_mma_peak(kind, 256, iters=2000)
    assert lo < t < hi, t


@pytest.mark.parametrize("M,N,K", [(2560, 4096, 512), (1100, 9728, 384)])
def test_ptpc_full_tile_several_tiles_per_cta(M, N, K):
    """More output tiles than 2 x SMs: every CTA runs 2-3 tiles, so the
    FP8 full-tile kernel's two TMEM accumulators both cycle (the epilogue of
    one tile runs beside the MMAs of the next)."""
    sm = torch.cuda.get_device_properties(dev()).multi_processor_count
    plan = mx.mxg_plan_gemm(mx.KIND_PTPC, M, N, K, sm, variant="full")
    assert plan["tiles"] > 2 * plan["ctas"]
    x, w = quant_pair(M, N, K, seed=M + N)
    y32 = run_ptpc(x, w, "full").cpu().numpy()
    rng = np.random.default_rng(M)
    rows = np.unique(np.concatenate([np.arange(0, M, 128), [M - 1], rng.choice(M, 40, replace=False)]))
    ref, bound = oracle_ptpc(x, w, rows=rows)
    assert_gemm_close(y32[rows], ref, bound, f"ptpc full {M}x{N}x{K}")
    y16 = run_ptpc(x, w, "full", out_f32=False)
    assert_codes_equal(y16.view(torch.int16).cpu().numpy().view(np.uint16), bf16_rne(y32),
                       "bf16 output = RNE(fp32 output)")


def test_ptpc_full_tile_banded_raster():
    """Operands far above L2 (157 MB of activations, 64 MB of weights): the
    full-tile GEMM walks its tiles in bands of token tiles whose activations
    take at most 32 MiB, here 19 token tiles (the last one ragged) in bands of
    4 + 4 + 4 + 4 + 3; sampled rows from every band, on both sides of each
    band boundary, match the oracle."""
    M, N, K = 2400, 1024, 65536
    x, w = quant_pair(M, N, K, seed=77)
    y32 = run_ptpc(x, w, "full").cpu().numpy()
    rows = np.array([0, 127, 128, 511, 512, 1023, 1024, 1151, 1535, 1536, 2047, 2048, 2200, 2303, 2304, 2399])
    ref, bound = oracle_ptpc(x, w, rows=rows)
    assert_gemm_close(y32[rows], ref, bound, f"ptpc full banded {M}x{N}x{K}")


@pytest.mark.parametrize("variant", ["full", "splitk"])
@pytest.mark.parametrize("kind", [0, 1])
def test_nonfinite_activation_rows_through_the_gemm(kind, variant):
    """A block (MXFP4) or a row (FP8) that holds a NaN or an infinity gets a
    NaN scale and zero codes (the OCP MX rule that a NaN scale makes the
    whole block NaN; the same reading for the per-token FP8 scale).  Its
    output row is then NaN in every column, and every other row is as usual:
    the NaN pattern and the finite values must match the oracle."""
    M, N, K = 40, 512, 1024
    x, w = quant_pair(M, N, K, seed=91)
    x = x.clone()
    x[3, 100] = float("nan")
    x[17, K - 1] = float("inf")
    x[30, 0] = float("-inf")
    if kind == 0:
        ref, bound = oracle_a4w4(x, w)
        for fused in (True, False):
            y = run_a4w4(x, w, variant, fused=fused).cpu().numpy()
            assert_gemm_close(y, ref, bound, f"a4w4 {variant} fused={fused} non-finite rows")
    else:
        ref, bound = oracle_ptpc(x, w)
        y = run_ptpc(x, w, variant).cpu().numpy()
        assert_gemm_close(y, ref, bound, f"ptpc {variant} non-finite rows")
    assert np.isnan(ref[[3, 17, 30]]).all() and not np.isnan(np.delete(ref, [3, 17, 30], axis=0)).any()
