"""Mutation check of the oracle's pins: plant a plausible mistake in a copy of
the oracle source (a wrong table entry, a flipped tie rule, a dropped sign,
swapped nibbles, a dropped scale term, a wrong exponent offset ...), build
it, and require that the pin suite fails against it.  Runs on the CPU only.
"""
import os
import subprocess
import sys
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "mxoracle.c")
PINS = ["tests/test_oracle_formats.py", "tests/test_oracle_quant.py", "tests/test_oracle_gemm.py",
        "tests/test_oracle_swiglu.py"]

MUTANTS = {
    "e2m1_table_entry": ("{0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0}", "{0.0, 0.5, 1.0, 1.5, 2.0, 2.5, 4.0, 6.0}"),
    "e2m1_tie_to_odd": ("if (d < best_d || (d == best_d && (c & 1u) == 0u && (best & 1u) != 0u)) {\n            best = c;\n            best_d = d;\n        }\n    }\n    return (uint8_t)(best | (signbit(v) ? 8u : 0u));",
                        "if (d < best_d || (d == best_d && (c & 1u) != 0u)) {\n            best = c;\n            best_d = d;\n        }\n    }\n    return (uint8_t)(best | (signbit(v) ? 8u : 0u));"),
    "e2m1_sign_dropped": ("return (uint8_t)(best | (signbit(v) ? 8u : 0u));", "return (uint8_t)(best | ((v < 0) ? 8u : 0u));"),
    "mx_emax_off_by_one": ("e = orc_floor_log2(amax) - 2;", "e = orc_floor_log2(amax) - 1;"),
    "mx_nibbles_swapped": ("(uint8_t)((c32[2 * j] & 0xFu) | ((c32[2 * j + 1] & 0xFu) << 4));", "(uint8_t)((c32[2 * j + 1] & 0xFu) | ((c32[2 * j] & 0xFu) << 4));"),
    "mx_zero_block_scale": ("e = -127; /* R1", "e = 0; /* R1"),
    "e4m3_subnormal_exp": ("mag = ldexp((double)m / 8.0, -6);", "mag = ldexp((double)m / 8.0, -7);"),
    "fp8_scale_constant": ("amax / 448.0f", "amax / 440.0f"),
    "fp8_reciprocal_multiply": ("orc_bf16_to_f32(xr[k]) / sv;", "orc_bf16_to_f32(xr[k]) * (1.0f / sv);"),
    "a4w4_scale_dropped": ("acc += blk * s;", "acc += blk;"),
    "a4w4_wrong_weight_scale_row": ("orc_e8m0_value(w_sf[(size_t)n * G + g]);", "orc_e8m0_value(w_sf[(size_t)n * G + (G - 1 - g)]);"),
    "ptpc_channel_scale_dropped": ("acc * (double)sa[m] * (double)sw[n];", "acc * (double)sa[m];"),
    "ptpc_bound_signed": ("accabs += fabs(p);", "accabs += p;"),
    "swiglu_gate_up_swapped": ("float g = orc_bf16_to_f32(row[j]);\n            float u = orc_bf16_to_f32(row[I + j]);",
                               "float g = orc_bf16_to_f32(row[I + j]);\n            float u = orc_bf16_to_f32(row[j]);"),
    "silu_exp_sign": ("float e = orc_exp_f32(-g);", "float e = orc_exp_f32(g);"),
    "silu_one_dropped": ("float d = 1.0f + e;", "float d = 0.5f + e;"),
    "exp_taylor_term_dropped": ("p = fmaf(p, r, c6);", "p = fmaf(p, r, 0.0f * c6);"),
    "exp_reduction_low_part_sign": ("r = r - nf * L2;", "r = r + nf * L2;"),
    "bf16_round_truncates": ("u += 0x7FFFu + ((u >> 16) & 1u);", "u += 0u * ((u >> 16) & 1u);"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor not unique/found: {name}"
    mut = tmp_path / "mut.c"
    mut.write_text(src.replace(old, new))
    so = tmp_path / "libmut.so"
    subprocess.run(["gcc", "-std=c11", "-O2", "-fopenmp", "-ffp-contract=off", "-fPIC",
                    "-shared", str(mut), "-o", str(so), "-lm"], check=True)
    env = dict(os.environ, MXORACLE_LIB=str(so))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider", *PINS],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"pins did not catch mutant {name}:\n{r.stdout[-2000:]}"
