"""GPU quantizers vs the CPU oracle: codes and scales must be bit-exact.

MXFP4: "Kimi-K3 DSpark O-Proj-only MXFP4", "Exact quantization coverage"
(E2M1 codes, E8M0 scale per 32 consecutive input channels; weight
(7168, 8192) with scale (7168, 256); dynamic MXFP4 activations).
FP8: "Kimi-K3-DSpark-FP8-PTPC", "Phase 1 FP8 PTPC Quantization".
"""
import numpy as np
import pytest
import torch

import fp8_block_scaled_dynamic_gb300 as mx
import oracle
import synth
from gpu_util import assert_codes_equal, dev, np_u8, untile_rows

pytestmark = pytest.mark.gpu


def bits_to_bf16(bits):
    return torch.from_numpy(np.asarray(bits, dtype=np.uint16).view(np.int16)).view(torch.bfloat16)


def check_mx(x_cpu, layout=mx.SF_SWIZZLED, what="mx"):
    d = dev()
    rows, K = x_cpu.shape
    if layout == mx.SF_SWIZZLED:
        codes, sf = mx.mx_quantize_act(x_cpu.to(d))
    else:
        codes, sf = mx.mx_quantize_weight(x_cpu.to(d), layout=layout)
    c_ref, s_ref = oracle.mx_quantize_rows(x_cpu)
    assert_codes_equal(np_u8(codes), c_ref, what + " codes")
    if layout == mx.SF_SWIZZLED:
        flat = np_u8(sf)
        assert flat.size == oracle.sf_swizzled_bytes(rows, K // 32)
        assert_codes_equal(oracle.sf_unswizzle(flat, rows, K // 32), s_ref, what + " scales")
        assert_codes_equal(flat, oracle.sf_swizzle(s_ref, pad_value=0), what + " scales incl. padding")
    else:
        assert_codes_equal(np_u8(sf), s_ref, what + " scales")


def test_mx_every_bf16_below_8_at_unit_scale():
    # each block: an anchor 7.9375 (fixes e = 0) + 31 values; all bf16 |v| < 8, both signs
    vals = np.concatenate([np.arange(0x0000, 0x40FF, dtype=np.uint16),
                           np.arange(0x8000, 0xC0FF, dtype=np.uint16)])
    n_blocks = -(-len(vals) // 31)
    vals = np.concatenate([vals, np.zeros(n_blocks * 31 - len(vals), np.uint16)])
    blocks = np.concatenate([np.full((n_blocks, 1), 0x40FE, np.uint16), vals.reshape(n_blocks, 31)], 1)
    pad = (-blocks.size) % (32 * 128)
    flat = np.concatenate([blocks.reshape(-1), np.zeros(pad, np.uint16)])
    x = bits_to_bf16(flat.reshape(-1, 128))
    check_mx(x, what="all bf16 < 8")


@pytest.mark.parametrize("shift", [-133, -127, -126, -100, -3, 5, 60, 120, 125])
def test_mx_power_of_two_shifted_values(shift):
    g = torch.Generator().manual_seed(abs(shift) + 17)
    x = (torch.randn(64, 512, generator=g) * 2.0 ** shift).to(torch.bfloat16)
    check_mx(x, what=f"shift {shift}")


def test_mx_special_values_and_nonfinite_blocks():
    rows = []
    sp = synth.special_values_bf16().view(torch.int16).numpy().view(np.uint16)
    rows.append(np.tile(sp, 4))
    r = np.full(128, 0x3F80, np.uint16)
    r[3] = 0x7FC0      # NaN -> block 0 gets scale 0xFF
    r[40] = 0x7F80     # +Inf -> block 1
    r[70] = 0xFF80     # -Inf -> block 2
    rows.append(r)
    rows.append(np.zeros(128, np.uint16))                   # zero blocks
    rows.append(np.full(128, 0x8000, np.uint16))            # -0 everywhere
    rows.append(np.array([0x0001, 0x8001, 0x007F] * 42 + [0, 0], np.uint16))  # subnormals
    x = bits_to_bf16(np.stack(rows))
    check_mx(x, what="special")


@pytest.mark.parametrize("M", [1, 7, 8, 9, 63, 64, 127, 129, 300])
def test_mx_act_ragged_rows(M):
    check_mx(synth.activation(M, 1024, seed=100 + M), what=f"M={M}")


def test_mx_act_strided_rows():
    d = dev()
    big = synth.activation(40, 1024 + 256, seed=5)
    x = big[:, :1024]
    codes, sf = mx.mx_quantize_act(big.to(d)[:, :1024])
    c_ref, s_ref = oracle.mx_quantize_rows(x.contiguous())
    assert_codes_equal(np_u8(codes), c_ref, "strided codes")
    assert_codes_equal(oracle.sf_unswizzle(np_u8(sf), 40, 32), s_ref, "strided scales")


@pytest.mark.parametrize("K", [128, 384, 7168])
def test_mx_weight_rowmajor_layout(K):
    check_mx(synth.weight(200, K, seed=K), layout=mx.SF_ROWMAJOR, what=f"rowmajor K={K}")


def test_mx_oproj_weight_full_size():
    # the stored o_proj weight of "Exact quantization coverage": (7168, 8192), scale (7168, 256)
    w = synth.weight(synth.OPROJ_N, synth.OPROJ_K, seed=synth.SEED_CFG0_W)
    d = dev()
    codes, sf = mx.mx_quantize_weight(w.to(d), layout=mx.SF_ROWMAJOR)
    assert tuple(codes.shape) == (7168, 4096) and tuple(sf.shape) == (7168, 256)
    c_ref, s_ref = oracle.mx_quantize_rows(w)
    assert_codes_equal(np_u8(codes), c_ref, "o_proj codes")
    assert_codes_equal(np_u8(sf), s_ref, "o_proj scales")
    _, sfz = mx.mx_quantize_weight(w.to(d), layout=mx.SF_SWIZZLED)
    assert_codes_equal(np_u8(sfz), oracle.sf_swizzle(s_ref), "o_proj swizzled scales")


@pytest.mark.parametrize("M,K", [(600, 10240), (520, 16384)])
def test_mx_act_rows_in_parts(M, K):
    """More than 512 rows of more than 8192 values: several CTAs stream
    parts of each row through shared memory (K = 10240: a 1024-chunk part
    and a 256-chunk one), padding rows of the swizzled scales included."""
    check_mx(synth.activation(M, K, seed=M + K, row_scale=True), what=f"parts {M}x{K}")


def test_mx_act_prefill_full_size():
    # 8 requests x 1024 tokens, per-row log-uniform scale in [0.1, 10], 0.1% x50 outliers
    x = synth.activation(8192, synth.OPROJ_K, seed=synth.act_seed(2, 0, 0), row_scale=True)
    check_mx(x, what="prefill act")


# ------------------------------------------------------------------ FP8
def check_fp8(x_cpu, what, rows=None):
    d = dev()
    q, s = mx.fp8_quantize_act(x_cpu.to(d))
    q = np_u8(q)
    s = s.cpu().numpy()
    if rows is not None:
        x_cpu = x_cpu[rows]
        q, s = q[rows], s[rows]
    q_ref, s_ref = oracle.fp8_quantize_rows(x_cpu.contiguous())
    assert_codes_equal(s.view(np.uint32), s_ref.view(np.uint32), what + " scales")
    assert_codes_equal(q, q_ref, what + " codes")


def test_fp8_every_bf16_at_unit_scale():
    # rows with amax exactly 448 (s = 1) holding every finite bf16 value below 448
    vals = np.arange(0, 0x43E0, dtype=np.uint16)  # 0x43E0 = 448.0
    vals = np.concatenate([vals, vals | 0x8000])
    per_row = 1023
    n = -(-len(vals) // per_row)
    vals = np.concatenate([vals, np.zeros(n * per_row - len(vals), np.uint16)]).reshape(n, per_row)
    x = np.concatenate([np.full((n, 1), 0x43E0, np.uint16), vals], 1)
    check_fp8(bits_to_bf16(x), "all bf16 at s=1")


@pytest.mark.parametrize("shift", [-130, -60, -8, 0, 9, 100])
def test_fp8_scaled_rows(shift):
    g = torch.Generator().manual_seed(shift + 1000)
    x = (torch.randn(33, 2048, generator=g) * 2.0 ** shift).to(torch.bfloat16)
    check_fp8(x, f"shift {shift}")


def test_fp8_special_rows():
    rows = [np.zeros(256, np.uint16), np.full(256, 0x8000, np.uint16)]
    r = np.full(256, 0x3F80, np.uint16); r[5] = 0x7FC0; rows.append(r)
    r = np.full(256, 0x3F80, np.uint16); r[9] = 0xFF80; rows.append(r)
    rows.append(np.tile(synth.special_values_bf16().view(torch.int16).numpy().view(np.uint16), 8))
    check_fp8(bits_to_bf16(np.stack(rows)), "special rows")


# rows from one to 30720 values, across the multiples of the 2048-value
# stride of the quantizer's 256 threads
@pytest.mark.parametrize("M,K", [(1, 128), (64, 7168), (3, 8192), (3, 8320), (64, 18432),
                                 (2, 24576), (2, 24704), (5, 30720)])
def test_fp8_act_shapes(M, K):
    check_fp8(synth.activation(M, K, seed=M * 7 + K), f"act {M}x{K}")


def staged_rows(M, K, seed):
    """More than 512 rows of K <= 8192 values (the quantizer that streams
    rows through shared memory): every finite bf16 value below 448 in rows
    whose first value is 448 (s = 1), then a zero row, an all -0 row, a row
    with a NaN and one with -Inf, then seeded activations."""
    vals = np.arange(0, 0x43E0, dtype=np.uint16)
    vals = np.concatenate([vals, vals | 0x8000])
    per_row = K - 1
    n = -(-len(vals) // per_row)
    vals = np.concatenate([vals, np.zeros(n * per_row - len(vals), np.uint16)]).reshape(n, per_row)
    ex = np.concatenate([np.full((n, 1), 0x43E0, np.uint16), vals], 1)
    special = np.zeros((4, K), np.uint16)
    special[1, :] = 0x8000
    special[2, :] = 0x3F80
    special[2, K // 3] = 0x7FC0
    special[3, :] = 0xBF80
    special[3, K - 1] = 0xFF80
    rest = synth.activation(M - n - 4, K, seed=seed).view(torch.int16).numpy().view(np.uint16)
    x = np.concatenate([ex, special, rest])
    assert x.shape[0] == M > 512
    return bits_to_bf16(x)


@pytest.mark.parametrize("M,K", [(700, 256), (600, 7168)])
def test_fp8_rows_through_shared_memory(M, K):
    """Exhaustive values, special rows and ragged rows (K = 256: most of a
    CTA's threads lie past the row) on the shared-memory-staged quantizer,
    row-major and in token tiles."""
    x = staged_rows(M, K, seed=M + K)
    check_fp8(x, f"staged {M}x{K}")
    q_ref, s_ref = oracle.fp8_quantize_rows(x)
    for T in (64, 128):
        q, s = mx.fp8_quantize_act_tiled(x.to(dev()), T)
        rows = -(-M // T) * T
        assert_codes_equal(untile_rows(np_u8(q), rows, K, T)[:M], q_ref, f"staged tiles {T} codes")
        sc = s.cpu().numpy()
        assert_codes_equal(sc.view(np.uint32), s_ref.view(np.uint32), f"staged tiles {T} scales")


@pytest.mark.parametrize("K", [8320, 30720])
def test_fp8_special_rows_long(K):
    """NaN / Inf rows, zero rows and all -0 rows in long rows."""
    base = synth.activation(6, K, seed=K).view(torch.int16).numpy().view(np.uint16).copy()
    base[1, :] = 0
    base[2, 17] = 0x7FC0          # NaN
    base[3, K - 1] = 0xFF80       # -Inf
    base[4, :] = 0x8000           # all -0
    check_fp8(bits_to_bf16(base), f"special rows K={K}")


def test_fp8_gate_up_weight_full_size_sampled_rows():
    # gate_up weight (2 x 18432, 7168): whole tensor on the GPU, 384 rows checked
    w = synth.weight(2 * synth.MLP_I, 7168, seed=synth.SEED_CFG3_GATE_UP)
    rows = np.sort(np.random.default_rng(0).choice(w.shape[0], 384, replace=False))
    check_fp8(w, "gate_up weight", rows=rows)


def test_fp8_prefill_act_sampled_rows():
    x = synth.activation(8192, 7168, seed=synth.act_seed(3, 0, 0))
    rows = np.sort(np.random.default_rng(1).choice(8192, 512, replace=False))
    check_fp8(x, "prefill act", rows=rows)
