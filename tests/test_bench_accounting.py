"""The algorithmic bytes bench.py divides by (roofline 'achieved' and the
value of every line), checked on the CPU against the library's own size
queries and the oracle's output shapes: one unit of work moves exactly its
operands once and its result once."""
import numpy as np
import pytest
import torch

import bench
import fp8_block_scaled_dynamic_gb300 as mx
import oracle


def test_oproj_decode_bytes_per_launch():
    # o_proj at M = 64: 29,360,128 weight code bytes + 1,835,008 scale bytes
    # + 262,144 activation code bytes + 16,384 activation scale bytes + 917,504 output bytes
    assert bench.a4w4_gemm_bytes(64, 7168, 8192) == 32_391_168


@pytest.mark.parametrize("M,N,K", [(64, 7168, 8192), (8, 7168, 8192), (8192, 7168, 8192), (300, 1024, 512)])
def test_a4w4_bytes_match_size_queries(M, N, K):
    want = (mx.mxg_weight_bytes(mx.KIND_A4W4, N, K, mx.SF_ROWMAJOR) + mx.mxg_sf_bytes(N, K, mx.SF_ROWMAJOR)
            + mx.mxg_weight_bytes(mx.KIND_A4W4, M, K, mx.SF_ROWMAJOR) + mx.mxg_sf_bytes(M, K, mx.SF_ROWMAJOR)
            + 2 * M * N)
    assert bench.a4w4_gemm_bytes(M, N, K) == want
    # bf16 activations in instead of codes and scales
    assert bench.a4w4_fused_bytes(M, N, K) == want - M * K // 2 - M * K // 32 + 2 * M * K


@pytest.mark.parametrize("M,N,K", [(64, 36864, 7168), (8192, 7168, 18432)])
def test_ptpc_bytes_match_size_queries(M, N, K):
    want = (mx.mxg_weight_bytes(mx.KIND_PTPC, N, K, mx.SF_ROWMAJOR) + 4 * N
            + mx.mxg_weight_bytes(mx.KIND_PTPC, M, K, mx.SF_ROWMAJOR) + 4 * M + 2 * M * N)
    assert bench.ptpc_gemm_bytes(M, N, K) == want


def test_quantizer_bytes_match_oracle_outputs():
    M, K = 6, 512
    x = torch.zeros(M, K, dtype=torch.bfloat16)
    codes, sf = oracle.mx_quantize_rows(x)
    assert bench.mx_quant_bytes(M, K) == x.numel() * 2 + np.asarray(codes).nbytes + np.asarray(sf).nbytes
    q, s = oracle.fp8_quantize_rows(x)
    assert bench.fp8_quant_bytes(M, K) == x.numel() * 2 + np.asarray(q).nbytes + np.asarray(s, np.float32).nbytes


def test_act_tile_rows_follow_the_plan():
    split = mx.mxg_plan_gemm(mx.KIND_A4W4, 64, 7168, 8192, 152)
    full = mx.mxg_plan_gemm(mx.KIND_A4W4, 8192, 7168, 8192, 152)
    assert split["variant"] == 2 and bench.act_tile_rows(split) == split["bn"] == 64
    assert full["variant"] == 1 and bench.act_tile_rows(full) == 128


@pytest.mark.parametrize("kind,M,N,K,kernels", [(0, 64, 7168, 8192, 2), (1, 64, 16384, 512, 1),
                                                 (1, 64, 12288, 1536, 1), (1, 64, 36864, 7168, 1),
                                                 (1, 64, 7168, 18432, 2)])
def test_launch_count_follows_the_plan(kind, M, N, K, kernels):
    """The bench's launch count: a GEMM call launches its kernel, plus the
    split-K reduce only when a tile's K is spread over several CTAs (not for
    whole-tile or full-tile plans)."""
    plan = mx.mxg_plan_gemm(kind, M, N, K, 152)
    assert bench.gemm_kernels(plan) == kernels
    assert ("stream-K" in bench.variant_desc(plan)) == (plan["variant"] == 2 and plan["seg_max"] > 1)


def test_bench_interval_check_catches_a_wrong_value():
    """The bf16 check the bench applies to its timed outputs rejects a value
    one bf16 step off when the tolerance is far below a step."""
    ref = np.array([[1.0, -3.0, 100.0]])
    bound = np.array([[1.0, 1.0, 1.0]])
    good = torch.tensor(ref, dtype=torch.float32).to(torch.bfloat16)
    assert bench.bf16_interval_check(good, ref, bound)[0]
    bad = good.clone()
    bad.view(torch.int16)[0, 2] += 1
    assert not bench.bf16_interval_check(bad, ref, bound)[0]
    nan_ref = np.array([[np.nan]])
    assert bench.bf16_interval_check(torch.tensor([[float("nan")]]).to(torch.bfloat16), nan_ref, bound[:, :1])[0]
    assert not bench.bf16_interval_check(torch.tensor([[0.0]]).to(torch.bfloat16), nan_ref, bound[:, :1])[0]
