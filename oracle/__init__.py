"""CPU oracle for the MXFP4 A4W4 / FP8 PTPC A8W8 path -- test infrastructure.

This package is the independent statement of what the CUDA library must
compute: a plain, slow C implementation (``mxoracle.c``) of OCP-MX E2M1/E8M0
and OCP E4M3 quantization and of the dequantize -> exact-accumulate GEMM,
plus numpy marshalling.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import it; the library never does, and the
two share no code.

Every function cites the passage it follows (page title and section):
  * "Kimi-K3 DSpark O-Proj-only MXFP4", "Exact quantization coverage":
    MXFP4 E2M1 codes + E8M0 scale per 32 consecutive input channels, stored
    weight (7168, 8192) and scale (7168, 256), dynamic MXFP4 activations,
    FP8 E4M3 per-output-channel weights with dynamic per-token activations.
  * "Kimi-K3-DSpark-FP8-PTPC", "Phase 1 FP8 PTPC Quantization": E4M3 weights,
    FP32 (out_features, 1) scales, dynamic per-token activation scales.
  * "Kimi-K3-Quark-MXFP4-AttnFP8", "Model Overview": "OCP MXFP4", "PTPC-FP8".

Parity status per function (what pins it; tests/test_oracle_formats.py,
test_oracle_quant.py, test_oracle_gemm.py, test_oracle_mutants.py):
  e2m1/e8m0/e4m3 decode   -- pinned (format tables, torch float8_e4m3fn)
  e2m1/e4m3 rounding      -- pinned (exhaustive bf16 scans vs exact rationals
                             and vs torch's float8_e4m3fn cast)
  mx_quantize_rows        -- pinned (closed-form cases, round-trip, scale
                             invariance, byte accounting of the pages)
  fp8_quantize_rows       -- pinned (amax = 448 row, power-of-two invariance)
  gemm_a4w4 / gemm_ptpc   -- pinned (exact rational brute force, integer
                             matmul special case)
  exp_f32 / silu_mul_f32  -- pinned (libm exp error bound over a dense scan,
                             scipy expit, the closed-form minimum of silu
                             via Lambert W, the identity silu(g) - silu(-g)
                             = g, saturation silu(g) = g for large g)
  swiglu_rows             -- pinned (gate/up order and bf16 rounding against
                             closed forms and torch's bf16 cast)
  gemm_a4w4_grouped       -- pinned (one-hot rows that only their own expert
                             can light, empty groups, one group = gemm_a4w4)
  sf_swizzle              -- bijection only; its placement is pinned on the
                             GPU by one-hot GEMMs (not from the pages)
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mxoracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libmxoracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile mxoracle.c with gcc (OpenMP, strict IEEE: no fast-math, no
    floating-point contraction).  Returns the shared-library path."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c11", "-O2", "-fopenmp", "-ffp-contract=off",
           "-fno-fast-math", "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    if _lib is None:
        # MXORACLE_LIB lets the mutation tests load a deliberately broken
        # copy of the oracle to show that the pins catch it.
        path = os.environ.get("MXORACLE_LIB") or build()
        L = ctypes.CDLL(path)
        u8p = ctypes.POINTER(ctypes.c_uint8)
        u16p = ctypes.POINTER(ctypes.c_uint16)
        f32p = ctypes.POINTER(ctypes.c_float)
        f64p = ctypes.POINTER(ctypes.c_double)
        i32p = ctypes.POINTER(ctypes.c_int)
        L.orc_bf16_to_f32.argtypes = [ctypes.c_uint16]
        L.orc_bf16_to_f32.restype = ctypes.c_float
        L.orc_e2m1_value.argtypes = [ctypes.c_uint8]
        L.orc_e2m1_value.restype = ctypes.c_double
        L.orc_e8m0_value.argtypes = [ctypes.c_uint8]
        L.orc_e8m0_value.restype = ctypes.c_double
        L.orc_e4m3_value.argtypes = [ctypes.c_uint8]
        L.orc_e4m3_value.restype = ctypes.c_double
        L.orc_e2m1_round.argtypes = [ctypes.c_double]
        L.orc_e2m1_round.restype = ctypes.c_uint8
        L.orc_e4m3_round.argtypes = [ctypes.c_float]
        L.orc_e4m3_round.restype = ctypes.c_uint8
        L.orc_floor_log2.argtypes = [ctypes.c_float]
        L.orc_floor_log2.restype = ctypes.c_int
        L.orc_mx_quantize_block.argtypes = [u16p, u8p, u8p]
        L.orc_mx_quantize_block.restype = None
        L.orc_mx_quantize_rows.argtypes = [u16p, ctypes.c_int, ctypes.c_int,
                                           ctypes.c_longlong, u8p, u8p]
        L.orc_mx_quantize_rows.restype = None
        L.orc_sf_swizzled_offset.argtypes = [ctypes.c_int] * 3
        L.orc_sf_swizzled_offset.restype = ctypes.c_size_t
        L.orc_sf_swizzled_bytes.argtypes = [ctypes.c_int] * 2
        L.orc_sf_swizzled_bytes.restype = ctypes.c_size_t
        L.orc_sf_swizzle.argtypes = [u8p, ctypes.c_int, ctypes.c_int, u8p]
        L.orc_sf_swizzle.restype = None
        L.orc_fp8_quantize_rows.argtypes = [u16p, ctypes.c_int, ctypes.c_int,
                                            ctypes.c_longlong, u8p, f32p]
        L.orc_fp8_quantize_rows.restype = None
        L.orc_gemm_a4w4.argtypes = [u8p, u8p, u8p, u8p, ctypes.c_int,
                                    ctypes.c_int, ctypes.c_int, i32p,
                                    ctypes.c_int, f64p, f64p]
        L.orc_gemm_a4w4.restype = None
        L.orc_gemm_ptpc.argtypes = [u8p, f32p, u8p, f32p, ctypes.c_int,
                                    ctypes.c_int, ctypes.c_int, i32p,
                                    ctypes.c_int, f64p, f64p]
        L.orc_gemm_ptpc.restype = None
        L.orc_exp_f32.argtypes = [ctypes.c_float]
        L.orc_exp_f32.restype = ctypes.c_float
        L.orc_silu_mul_f32.argtypes = [ctypes.c_float, ctypes.c_float]
        L.orc_silu_mul_f32.restype = ctypes.c_float
        L.orc_f32_to_bf16.argtypes = [ctypes.c_float]
        L.orc_f32_to_bf16.restype = ctypes.c_uint16
        L.orc_swiglu_rows.argtypes = [u16p, ctypes.c_int, ctypes.c_int, ctypes.c_longlong, u16p]
        L.orc_swiglu_rows.restype = None
        L.orc_num_threads.argtypes = []
        L.orc_num_threads.restype = ctypes.c_int
        _lib = L
    return _lib


def _ptr(a: np.ndarray, ctype):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _as_bf16_bits(x) -> np.ndarray:
    """Accept a torch bf16 tensor or a uint16 numpy array of bf16 bits."""
    if isinstance(x, np.ndarray):
        assert x.dtype == np.uint16
        return np.ascontiguousarray(x)
    import torch  # only for the bit reinterpretation of a CPU tensor
    assert x.dtype == torch.bfloat16
    return np.ascontiguousarray(x.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16))


# ---- scalar format helpers ------------------------------------------------
def e2m1_value(code: int) -> float:
    return lib().orc_e2m1_value(code)


def e8m0_value(c: int) -> float:
    return lib().orc_e8m0_value(c)


def e4m3_value(code: int) -> float:
    return lib().orc_e4m3_value(code)


def e2m1_round(v: float) -> int:
    return lib().orc_e2m1_round(v)


def e4m3_round(v: float) -> int:
    return lib().orc_e4m3_round(v)


def floor_log2(a: float) -> int:
    return lib().orc_floor_log2(a)


def bf16_to_f32(bits: int) -> float:
    return lib().orc_bf16_to_f32(bits)


# ---- quantizers -------------------------------------------------------------
def mx_quantize_block(x_bits: np.ndarray):
    """One OCP-MX block of 32 bf16 values -> (32 unpacked codes, scale code)."""
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    assert x.shape == (32,)
    codes = np.zeros(32, np.uint8)
    sc = np.zeros(1, np.uint8)
    lib().orc_mx_quantize_block(_ptr(x, ctypes.c_uint16), _ptr(codes, ctypes.c_uint8),
                                _ptr(sc, ctypes.c_uint8))
    return codes, int(sc[0])


def mx_quantize_rows(x):
    """x: (rows, K) bf16 -> (codes (rows, K/2) u8 packed, sf (rows, K/32) u8
    row-major, the stored layout of "Exact quantization coverage")."""
    xb = _as_bf16_bits(x)
    rows, K = xb.shape
    assert K % 32 == 0
    codes = np.zeros((rows, K // 2), np.uint8)
    sf = np.zeros((rows, K // 32), np.uint8)
    lib().orc_mx_quantize_rows(_ptr(xb, ctypes.c_uint16), rows, K, K,
                               _ptr(codes, ctypes.c_uint8), _ptr(sf, ctypes.c_uint8))
    return codes, sf


def sf_swizzled_offset(r: int, g: int, G: int) -> int:
    return lib().orc_sf_swizzled_offset(r, g, G)


def sf_swizzled_bytes(rows: int, G: int) -> int:
    return lib().orc_sf_swizzled_bytes(rows, G)


def sf_swizzle(sf_rowmajor: np.ndarray, pad_value: int = 0) -> np.ndarray:
    """Row-major (rows, G) scales -> flat 128x4-tile layout; padding bytes
    are filled with pad_value (their content is unspecified)."""
    sf = np.ascontiguousarray(sf_rowmajor, dtype=np.uint8)
    rows, G = sf.shape
    out = np.full(sf_swizzled_bytes(rows, G), pad_value, np.uint8)
    lib().orc_sf_swizzle(_ptr(sf, ctypes.c_uint8), rows, G, _ptr(out, ctypes.c_uint8))
    return out


def sf_unswizzle(sf_swz: np.ndarray, rows: int, G: int) -> np.ndarray:
    """Inverse of sf_swizzle on the valid region (rows, G)."""
    r = np.arange(rows)[:, None]
    g = np.arange(G)[None, :]
    off = ((r // 128) * (G // 4) + g // 4) * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + g % 4
    return np.asarray(sf_swz)[off]


def fp8_quantize_rows(x):
    """x: (rows, K) bf16 -> (q (rows, K) u8 E4M3 codes, s (rows,) f32)."""
    xb = _as_bf16_bits(x)
    rows, K = xb.shape
    q = np.zeros((rows, K), np.uint8)
    s = np.zeros(rows, np.float32)
    lib().orc_fp8_quantize_rows(_ptr(xb, ctypes.c_uint16), rows, K, K,
                                _ptr(q, ctypes.c_uint8), _ptr(s, ctypes.c_float))
    return q, s


# ---- reference GEMMs --------------------------------------------------------
def _rows_arg(M, rows):
    if rows is None:
        return None, M
    idx = np.ascontiguousarray(np.asarray(rows, dtype=np.int32))
    return idx, int(idx.size)


def gemm_a4w4(a_codes, a_sf, w_codes, w_sf, rows=None):
    """Reference y = x . W^T over dequantized MXFP4 operands (row-major
    scales).  Returns (ref, bound) as float64 arrays (len(rows) or M, N)."""
    a_codes = np.ascontiguousarray(a_codes, np.uint8)
    w_codes = np.ascontiguousarray(w_codes, np.uint8)
    a_sf = np.ascontiguousarray(a_sf, np.uint8)
    w_sf = np.ascontiguousarray(w_sf, np.uint8)
    M, K2 = a_codes.shape
    N = w_codes.shape[0]
    K = 2 * K2
    assert w_codes.shape == (N, K2) and a_sf.shape == (M, K // 32) and w_sf.shape == (N, K // 32)
    idx, nrows = _rows_arg(M, rows)
    ref = np.zeros((nrows, N), np.float64)
    bound = np.zeros((nrows, N), np.float64)
    lib().orc_gemm_a4w4(_ptr(a_codes, ctypes.c_uint8), _ptr(a_sf, ctypes.c_uint8),
                        _ptr(w_codes, ctypes.c_uint8), _ptr(w_sf, ctypes.c_uint8),
                        M, N, K, None if idx is None else _ptr(idx, ctypes.c_int),
                        nrows, _ptr(ref, ctypes.c_double), _ptr(bound, ctypes.c_double))
    return ref, bound


def gemm_ptpc(qa, sa, qw, sw, rows=None):
    """Reference y = (sum_k v(qa) v(qw)) * sa[m] * sw[n].  Returns (ref, bound)."""
    qa = np.ascontiguousarray(qa, np.uint8)
    qw = np.ascontiguousarray(qw, np.uint8)
    sa = np.ascontiguousarray(sa, np.float32).reshape(-1)
    sw = np.ascontiguousarray(sw, np.float32).reshape(-1)
    M, K = qa.shape
    N = qw.shape[0]
    assert qw.shape == (N, K) and sa.shape == (M,) and sw.shape == (N,)
    idx, nrows = _rows_arg(M, rows)
    ref = np.zeros((nrows, N), np.float64)
    bound = np.zeros((nrows, N), np.float64)
    lib().orc_gemm_ptpc(_ptr(qa, ctypes.c_uint8), _ptr(sa, ctypes.c_float),
                        _ptr(qw, ctypes.c_uint8), _ptr(sw, ctypes.c_float),
                        M, N, K, None if idx is None else _ptr(idx, ctypes.c_int),
                        nrows, _ptr(ref, ctypes.c_double), _ptr(bound, ctypes.c_double))
    return ref, bound


def gemm_a4w4_grouped(a_codes, a_sf, w_codes, w_sf, row_off):
    """Grouped (MoE) A4W4: the token rows arrive grouped by expert (rows
    row_off[e] .. row_off[e+1]-1 were routed to expert e; a group may be
    empty), and each group goes through its own expert's MXFP4 weight:
    y[rows of e] = x[rows of e] . W_e^T ("Kimi-K3-Quark-MXFP4-AttnFP8", "Model
    Overview": the experts are OCP MXFP4).  w_codes / w_sf: one (N, K/2) /
    (N, K/32) array per expert.  Returns (ref, bound) (M, N) float64.  The
    routing and the token permutation that produce the grouping are a
    dispatch step of their own, not part of the GEMM."""
    a_codes = np.ascontiguousarray(a_codes, np.uint8)
    a_sf = np.ascontiguousarray(a_sf, np.uint8)
    off = [int(v) for v in row_off]
    E = len(off) - 1
    assert len(w_codes) == E and len(w_sf) == E and off[0] == 0 and off[-1] == a_codes.shape[0]
    assert all(off[e] <= off[e + 1] for e in range(E))
    N = np.asarray(w_codes[0]).shape[0]
    ref = np.zeros((a_codes.shape[0], N), np.float64)
    bound = np.zeros((a_codes.shape[0], N), np.float64)
    for e in range(E):
        r0, r1 = off[e], off[e + 1]
        if r1 > r0:
            ref[r0:r1], bound[r0:r1] = gemm_a4w4(a_codes[r0:r1], a_sf[r0:r1], w_codes[e], w_sf[e])
    return ref, bound


# ---- SwiGLU between gate_up and down --------------------------------------
def exp_f32(t: float) -> float:
    """e^t in binary32 by the Cody-Waite method the SwiGLU uses (R17)."""
    return lib().orc_exp_f32(t)


def silu_mul_f32(g: float, u: float) -> float:
    """silu(g) * u in binary32, one IEEE operation at a time (R14, R17)."""
    return lib().orc_silu_mul_f32(g, u)


def f32_to_bf16(f: float) -> int:
    return lib().orc_f32_to_bf16(f)


def swiglu_rows(gu):
    """gu: (rows, 2I) bf16 gate_up output [gate | up] -> h (rows, I) as uint16
    bf16 bits, h = bf16(silu(gate) * up) (R14-R17)."""
    gb = _as_bf16_bits(gu)
    rows, I2 = gb.shape
    assert I2 % 2 == 0
    I = I2 // 2
    h = np.zeros((rows, I), np.uint16)
    lib().orc_swiglu_rows(_ptr(gb, ctypes.c_uint16), rows, I, I2, _ptr(h, ctypes.c_uint16))
    return h


def swiglu_fp8_quantize_rows(gu):
    """The fused step between gate_up and down: h = swiglu_rows(gu), then the
    per-token FP8 quantization of h.  Returns (h bits, q, s)."""
    h = swiglu_rows(gu)
    q, s = fp8_quantize_rows(h)
    return h, q, s


def num_threads() -> int:
    return lib().orc_num_threads()
