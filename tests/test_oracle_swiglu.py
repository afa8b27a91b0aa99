"""Pins of the oracle's SwiGLU step between the packed gate_up projection and
the down projection ("Kimi-K3-DSpark-FP8-PTPC", "Phase 1 FP8 PTPC
Quantization": gate_proj and up_proj packed into one gate_up_proj; the
activation itself is a reading, SwiGLU).  Nothing here retypes the oracle's
formula: the pins are a library exp and expit, closed forms of silu
(its minimum through Lambert W, silu(g) - silu(-g) = g, silu(g) = g once
e^-g vanishes next to 1), the gate/up order on values where the two orders
differ, and torch's bf16 rounding.
"""
import math

import numpy as np
import pytest
import torch

import oracle

scipy_special = pytest.importorskip("scipy.special")


def ulp32(x):
    x = np.abs(np.asarray(x, np.float64))
    return np.spacing(x.astype(np.float32)).astype(np.float64)


def f32_grid(lo, hi, n):
    return np.unique(np.linspace(lo, hi, n).astype(np.float32))


# ---------------------------------------------------------------- e^t
def test_exp_within_two_ulp_of_libm():
    """Cody-Waite reduction + Taylor series through r^7/7!: within 2 units in
    the last place of the correctly rounded binary32 e^t over the whole
    range the SwiGLU uses (a dense scan plus every power-of-two boundary
    of the reduction), measured against math.exp in binary64."""
    ts = np.concatenate([f32_grid(-87.2, 88.7, 200001),
                         (np.arange(-125, 128) * math.log(2)).astype(np.float32),
                         (np.arange(-125, 128) * math.log(2) + math.log(2) / 2).astype(np.float32)])
    got = np.array([oracle.exp_f32(float(t)) for t in ts], np.float64)
    want = np.exp(ts.astype(np.float64))
    err = np.abs(got - want) / ulp32(want)
    assert err.max() <= 2.0, (float(err.max()), float(ts[np.argmax(err)]))


def test_exp_special_values():
    assert oracle.exp_f32(0.0) == 1.0
    assert oracle.exp_f32(-0.0) == 1.0
    assert oracle.exp_f32(100.0) == math.inf
    assert oracle.exp_f32(-100.0) == 0.0
    assert math.isnan(oracle.exp_f32(math.nan))
    assert oracle.exp_f32(-math.inf) == 0.0 and oracle.exp_f32(math.inf) == math.inf
    # e^1 within one binary32 step of e
    assert abs(oracle.exp_f32(1.0) - math.e) <= float(np.spacing(np.float32(math.e)))


# ---------------------------------------------------------------- silu
def test_silu_against_expit():
    """silu(g) = g * expit(g) (scipy, binary64) within 3 binary32 steps."""
    gs = np.concatenate([f32_grid(-40.0, 40.0, 80001), f32_grid(-1e-3, 1e-3, 2001)])
    got = np.array([oracle.silu_mul_f32(float(g), 1.0) for g in gs], np.float64)
    want = gs.astype(np.float64) * scipy_special.expit(gs.astype(np.float64))
    tol = 3.0 * ulp32(want) + 1e-45
    bad = np.abs(got - want) > tol
    assert not bad.any(), (gs[bad][:5], got[bad][:5], want[bad][:5])


def test_silu_minimum_is_minus_lambert_w_of_one_over_e():
    """d/dx x sigma(x) = 0 at x* = -(1 + W(1/e)), where silu(x*) = -W(1/e)
    = -0.27846454276107...: the oracle's silu takes its smallest value next
    to x*, and that value is -W(1/e) to binary32 accuracy."""
    w = float(np.real(scipy_special.lambertw(1.0 / math.e)))
    x_star = -(1.0 + w)
    gs = f32_grid(x_star - 0.05, x_star + 0.05, 20001)
    vals = np.array([oracle.silu_mul_f32(float(g), 1.0) for g in gs])
    assert abs(float(vals.min()) - (-w)) <= 2 * float(np.spacing(np.float32(w)))
    # the minimum is flat: the argmin is within a few 1e-3 of x*
    assert abs(float(gs[np.argmin(vals)]) - x_star) < 5e-3


def test_silu_odd_part_is_identity():
    """sigma(g) + sigma(-g) = 1, so silu(g) - silu(-g) = g."""
    gs = f32_grid(0.0, 30.0, 30001)
    d = np.array([oracle.silu_mul_f32(float(g), 1.0) - oracle.silu_mul_f32(float(-g), 1.0) for g in gs])
    assert np.all(np.abs(d - gs.astype(np.float64)) <= 4 * ulp32(gs) + 1e-45)


def test_silu_saturates_and_special_cases():
    # e^-g < 2^-25 makes 1 + e^-g round to 1: silu(g) = g exactly
    for g in (17.5, 20.0, 100.0, 3.0e38):
        assert oracle.silu_mul_f32(g, 1.0) == np.float32(g)
    assert oracle.silu_mul_f32(0.0, 5.0) == 0.0
    assert oracle.silu_mul_f32(5.0, 0.0) == 0.0
    v = oracle.silu_mul_f32(-200.0, 1.0)  # -200 / inf
    assert v == 0.0 and math.copysign(1.0, v) == -1.0
    assert math.isnan(oracle.silu_mul_f32(math.nan, 1.0))
    assert math.isnan(oracle.silu_mul_f32(1.0, math.nan))
    assert oracle.silu_mul_f32(math.inf, 2.0) == math.inf
    assert math.isnan(oracle.silu_mul_f32(-math.inf, 1.0))  # -inf / inf


# ---------------------------------------------------------------- the row step
def bf16(vals):
    return torch.tensor(vals, dtype=torch.float32).to(torch.bfloat16)


def test_gate_is_the_first_half_of_the_row():
    """[gate | up]: with gate = 20 (silu(20) = 20) and up = 3, h = 60; the
    swapped order would give silu(3) * 20 = 57.15..."""
    I = 4
    gu = bf16([[20.0, 20.0, 0.0, -200.0, 3.0, 1.0, 7.0, 2.0]])
    h = oracle.swiglu_rows(gu)
    hv = torch.from_numpy(h.view(np.int16)).view(torch.bfloat16).float().numpy()
    assert hv.shape == (1, I)
    assert hv[0, 0] == 60.0 and hv[0, 1] == 20.0 and hv[0, 2] == 0.0
    assert hv[0, 3] == 0.0 and math.copysign(1.0, hv[0, 3]) == -1.0  # silu(-200) * 2: -200 / inf = -0


def test_h_is_bf16_round_to_nearest_even_of_the_binary32_product():
    """The bf16 rounding of h equals torch's bf16 cast of the binary32
    silu(g) * u (a library rounding), row by row, over random gate_up rows."""
    g = torch.Generator().manual_seed(5)
    gu = (torch.randn(6, 2 * 512, generator=g) * 3).to(torch.bfloat16)
    h = oracle.swiglu_rows(gu)
    f = gu.float().numpy()
    prod = np.array([[oracle.silu_mul_f32(float(f[r, j]), float(f[r, 512 + j])) for j in range(512)]
                     for r in range(6)], np.float32)
    want = torch.from_numpy(prod).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert (h == want).all()
    # and h is within a bf16 half step (plus binary32 error) of the binary64 definition
    g64, u64 = f[:, :512].astype(np.float64), f[:, 512:].astype(np.float64)
    exact = g64 * scipy_special.expit(g64) * u64
    hv = torch.from_numpy(h.view(np.int16)).view(torch.bfloat16).double().numpy()
    assert np.all(np.abs(hv - exact) <= np.abs(exact) * (2.0 ** -8 + 2.0 ** -21) + 1e-30)


def test_swiglu_quantization_is_the_per_token_fp8_of_h():
    """The fused step's codes and scale are the per-token FP8 quantization of
    h: the row's scale is amax(h) / 448 and the largest |h| maps to 448."""
    g = torch.Generator().manual_seed(9)
    gu = torch.randn(3, 2 * 256, generator=g).to(torch.bfloat16)
    h, q, s = oracle.swiglu_fp8_quantize_rows(gu)
    hv = torch.from_numpy(h.view(np.int16)).view(torch.bfloat16).float().numpy()
    for r in range(3):
        amax = np.float32(np.abs(hv[r]).max())
        assert s[r] == np.float32(amax / np.float32(448.0))
        j = int(np.argmax(np.abs(hv[r])))
        assert abs(oracle.e4m3_value(int(q[r, j]))) == 448.0
