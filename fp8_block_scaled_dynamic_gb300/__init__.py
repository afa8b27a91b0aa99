"""GB300 (sm_103a) MXFP4 A4W4 / FP8 PTPC A8W8 library -- Python binding.

Argument marshalling only: every function below takes torch tensors, checks
dtypes and shapes, allocates outputs with torch (device memory is the only
thing torch provides here) and calls the entry point of the same name in
``libmxgemm.so`` (C ABI, ``include/mxgemm.h``).  All arithmetic runs in the
library's CUDA kernels; there is no CPU or PyTorch fallback -- if the
library is missing, importing a function raises.

The quantized formats follow page "Kimi-K3 DSpark O-Proj-only MXFP4", section
"Exact quantization coverage" (MXFP4: E2M1 codes, E8M0 scale per 32
consecutive input channels) and page "Kimi-K3-DSpark-FP8-PTPC", section
"Phase 1 FP8 PTPC Quantization" (E4M3, per-output-channel FP32 scale,
dynamic per-token activation scale).
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmxgemm.so")

MXG_OK = 0
STATUS_NAMES = {0: "MXG_OK", 1: "MXG_ERR_INVALID_ARG", 2: "MXG_ERR_UNSUPPORTED_SHAPE",
                3: "MXG_ERR_MISALIGNED", 4: "MXG_ERR_UNSUPPORTED_DEVICE", 5: "MXG_ERR_CUDA",
                6: "MXG_ERR_TIMEOUT", 7: "MXG_ERR_WORKSPACE"}
SF_ROWMAJOR, SF_SWIZZLED, TILED, PANEL = 0, 1, 2, 3
TILE_BYTES = 16384
PANEL_ROWS = 256
# weights_tiled values of the GEMM calls: the weight codes' layout
W_ROWMAJOR, W_TILED, W_PANEL = 0, 1, 2
OUT_BF16, OUT_F32 = 0, 1
VARIANTS = {"auto": 0, "full": 1, "splitk": 2}
KIND_A4W4, KIND_PTPC = 0, 1


class MxgError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} failed: {STATUS_NAMES.get(status, status)}")


class GemmOpts(ctypes.Structure):
    _fields_ = [("variant", ctypes.c_int), ("ctas", ctypes.c_int),
                ("workspace", ctypes.c_void_p), ("ws_bytes", ctypes.c_size_t),
                ("dev_status", ctypes.c_void_p), ("timeout_ms", ctypes.c_uint32),
                ("debug_stall", ctypes.c_int), ("weights_static", ctypes.c_int),
                ("weights_tiled", ctypes.c_int), ("act_tile_rows", ctypes.c_int),
                ("trace", ctypes.c_void_p), ("splitk_reduce", ctypes.c_int), ("cta_pair", ctypes.c_int)]


REDUCE = {"default": 0, "kernel": 1}


class Plan(ctypes.Structure):
    _fields_ = [("variant", ctypes.c_int), ("bm", ctypes.c_int), ("bn", ctypes.c_int),
                ("ctas", ctypes.c_int), ("tiles", ctypes.c_int), ("kblocks", ctypes.c_int),
                ("seg_max", ctypes.c_int), ("ws_bytes", ctypes.c_size_t), ("cta_pair", ctypes.c_int)]


_lib = None
_lib_lock = threading.Lock()


def lib() -> ctypes.CDLL:
    """The loaded C library.  Raises if it has not been built."""
    global _lib
    with _lib_lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is missing: build it with "
                    "`python -c 'import __graft_entry__ as g; g.build()'` (there is no fallback)")
            L = ctypes.CDLL(LIB_PATH)
            vp, i, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
            L.mxg_sf_bytes.argtypes = [i, i, i]
            L.mxg_sf_bytes.restype = sz
            L.mxg_plan_gemm.argtypes = [i, i, i, i, i, ctypes.POINTER(GemmOpts), ctypes.POINTER(Plan)]
            L.mxg_plan_gemm.restype = i
            L.mxg_gemm_workspace_bytes.argtypes = [i, i, i, i, i, ctypes.POINTER(GemmOpts)]
            L.mxg_gemm_workspace_bytes.restype = sz
            L.mx_quantize_weight.argtypes = [vp, i, i, i, vp, vp, i, vp]
            L.mx_quantize_weight.restype = i
            L.mx_quantize_act.argtypes = [vp, i, i, i, vp, vp, vp]
            L.mx_quantize_act.restype = i
            L.mx_gemm_a4w4.argtypes = [vp, vp, vp, i, vp, vp, i, i, i, vp, i, i,
                                       ctypes.POINTER(GemmOpts), vp]
            L.mx_gemm_a4w4.restype = i
            L.fp8_quantize_act.argtypes = [vp, i, i, i, vp, vp, vp]
            L.fp8_quantize_act.restype = i
            L.fp8_quantize_weight.argtypes = [vp, i, i, i, vp, vp, i, vp]
            L.fp8_quantize_weight.restype = i
            L.mxg_weight_bytes.argtypes = [i, i, i, i]
            L.mxg_weight_bytes.restype = sz
            L.mxg_act_tiled_bytes.argtypes = [i, i, i, i]
            L.mxg_act_tiled_bytes.restype = sz
            L.mx_quantize_act_tiled.argtypes = [vp, i, i, i, i, vp, vp, vp]
            L.mx_quantize_act_tiled.restype = i
            L.fp8_quantize_act_tiled.argtypes = [vp, i, i, i, i, vp, vp, vp]
            L.fp8_quantize_act_tiled.restype = i
            L.swiglu_fp8_quantize.argtypes = [vp, i, i, i, i, vp, vp, vp, i, vp]
            L.swiglu_fp8_quantize.restype = i
            L.fp8_gemm_ptpc.argtypes = [vp, vp, vp, vp, i, i, i, vp, i, i,
                                        ctypes.POINTER(GemmOpts), vp]
            L.fp8_gemm_ptpc.restype = i
            L.mxg_grouped_workspace_bytes.argtypes = [i, i, i]
            L.mxg_grouped_workspace_bytes.restype = sz
            L.mx_gemm_a4w4_grouped.argtypes = [vp, i, vp, i, vp, i, i, i, vp, i, i,
                                               ctypes.POINTER(GemmOpts), vp]
            L.mx_gemm_a4w4_grouped.restype = i
            L.mxg_mma_peak.argtypes = [i, i, i, ctypes.POINTER(ctypes.c_double), vp]
            L.mxg_mma_peak.restype = i
            L.mxg_query_status.argtypes = [vp, vp]
            L.mxg_query_status.restype = i
            L.mxg_status_string.argtypes = [i]
            L.mxg_status_string.restype = ctypes.c_char_p
            _lib = L
    return _lib


def _check(fn: str, st: int):
    if st != MXG_OK:
        raise MxgError(fn, st)


def _stream(stream=None) -> ctypes.c_void_p:
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t) -> ctypes.c_void_p:
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


def _need(cond: bool, msg: str):
    if not cond:
        raise ValueError(msg)


# ---------------------------------------------------------------- sizes / plan
def mxg_sf_bytes(rows: int, K: int, layout: int = SF_SWIZZLED) -> int:
    return int(lib().mxg_sf_bytes(rows, K, layout))


def mxg_weight_bytes(kind: int, N: int, K: int, layout: int) -> int:
    return int(lib().mxg_weight_bytes(kind, N, K, layout))


def mxg_plan_gemm(kind: int, M: int, N: int, K: int, sm_count: int,
                  variant: str = "auto", ctas: int = 0, splitk_reduce: str = "default",
                  cta_pair: bool = False) -> dict:
    """Pure host dispatcher: the variant/tile/grid/workspace of a GEMM."""
    o = GemmOpts(variant=VARIANTS[variant], ctas=ctas, splitk_reduce=REDUCE[splitk_reduce], cta_pair=int(cta_pair))
    p = Plan()
    _check("mxg_plan_gemm", lib().mxg_plan_gemm(kind, M, N, K, sm_count, ctypes.byref(o), ctypes.byref(p)))
    return {f: getattr(p, f) for f, _ in Plan._fields_}


def mxg_gemm_workspace_bytes(kind: int, fused: bool, M: int, N: int, K: int,
                             variant: str = "auto", ctas: int = 0, splitk_reduce: str = "default") -> int:
    o = GemmOpts(variant=VARIANTS[variant], ctas=ctas, splitk_reduce=REDUCE[splitk_reduce])
    return int(lib().mxg_gemm_workspace_bytes(kind, int(fused), M, N, K, ctypes.byref(o)))


_ws_cache: dict = {}


def workspace(nbytes: int, device=None) -> torch.Tensor | None:
    """A zero-filled device workspace of at least nbytes, cached per device.
    It is reused across calls on one stream; give concurrent streams their
    own workspace."""
    if nbytes <= 0:
        return None
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    cur = _ws_cache.get(dev)
    if cur is None or cur.numel() < nbytes:
        cur = torch.zeros(max(nbytes, 1 << 20), dtype=torch.uint8, device=dev)
        _ws_cache[dev] = cur
    return cur


# ---------------------------------------------------------------- quantizers
def mx_quantize_weight(w: torch.Tensor, layout: int = SF_SWIZZLED, codes=None, sf=None, stream=None):
    """Offline MXFP4 weight conversion: w (N, K) bf16 -> (codes u8, sf u8).
    layout SF_ROWMAJOR: codes (N, K/2), sf (N, K/32); SF_SWIZZLED: codes
    (N, K/2), sf flat 128x4 tiles; TILED: codes in 16 KiB weight tiles
    (shape (N, K/2) bytes, tile-ordered), sf flat 128x4 tiles; PANEL: codes
    flat (mxg_weight_bytes bytes) in 256-row panels holding the scales too,
    sf None."""
    _need(w.is_cuda and w.dtype == torch.bfloat16 and w.dim() == 2 and w.stride(1) == 1,
          "w must be a CUDA bf16 (N, K) tensor with unit inner stride")
    N, K = w.shape
    if layout == PANEL:
        if codes is None:
            nbytes = mxg_weight_bytes(KIND_A4W4, N, K, PANEL)
            _need(nbytes > 0, "the panel layout needs K % 256 == 0")
            codes = torch.empty(nbytes, dtype=torch.uint8, device=w.device)
        _check("mx_quantize_weight", lib().mx_quantize_weight(
            _ptr(w), N, K, w.stride(0), _ptr(codes), None, layout, _stream(stream)))
        return codes, None
    if codes is None:
        codes = torch.empty(N, K // 2, dtype=torch.uint8, device=w.device)
    if sf is None:
        shape = (N, K // 32) if layout == SF_ROWMAJOR else (mxg_sf_bytes(N, K, SF_SWIZZLED),)
        sf = torch.empty(shape, dtype=torch.uint8, device=w.device)
    _check("mx_quantize_weight", lib().mx_quantize_weight(
        _ptr(w), N, K, w.stride(0), _ptr(codes), _ptr(sf), layout, _stream(stream)))
    return codes, sf


def mx_quantize_act(x: torch.Tensor, codes=None, sf=None, stream=None):
    """Dynamic MXFP4 activation quantization: x (M, K) bf16 -> (codes (M, K/2),
    sf swizzled flat, padding rows zero)."""
    _need(x.is_cuda and x.dtype == torch.bfloat16 and x.dim() == 2 and x.stride(1) == 1,
          "x must be a CUDA bf16 (M, K) tensor with unit inner stride")
    M, K = x.shape
    if codes is None:
        codes = torch.empty(M, K // 2, dtype=torch.uint8, device=x.device)
    if sf is None:
        sf = torch.empty(mxg_sf_bytes(M, K, SF_SWIZZLED), dtype=torch.uint8, device=x.device)
    _check("mx_quantize_act", lib().mx_quantize_act(
        _ptr(x), M, K, x.stride(0), _ptr(codes), _ptr(sf), _stream(stream)))
    return codes, sf


def fp8_quantize_weight(w: torch.Tensor, layout: int = SF_ROWMAJOR, q=None, scale=None, stream=None):
    """Per-output-channel E4M3 weight conversion: w (N, K) bf16 -> (q (N, K)
    bytes, row-major or in 16 KiB weight tiles (layout TILED), or flat in
    256-row panels (layout PANEL, mxg_weight_bytes bytes), scale (N,) f32)."""
    _need(w.is_cuda and w.dtype == torch.bfloat16 and w.dim() == 2 and w.stride(1) == 1,
          "w must be a CUDA bf16 (N, K) tensor with unit inner stride")
    N, K = w.shape
    if q is None:
        q = (torch.empty(mxg_weight_bytes(KIND_PTPC, N, K, PANEL), dtype=torch.uint8, device=w.device)
             if layout == PANEL else torch.empty(N, K, dtype=torch.uint8, device=w.device))
    if scale is None:
        scale = torch.empty(N, dtype=torch.float32, device=w.device)
    _check("fp8_quantize_weight", lib().fp8_quantize_weight(
        _ptr(w), N, K, w.stride(0), _ptr(q), _ptr(scale), layout, _stream(stream)))
    return q, scale


def mxg_act_tiled_bytes(kind: int, M: int, K: int, tile_rows: int) -> int:
    return int(lib().mxg_act_tiled_bytes(kind, M, K, tile_rows))


def mx_quantize_act_tiled(x: torch.Tensor, tile_rows: int, codes=None, sf=None, stream=None):
    """mx_quantize_act with the codes in the activation tile layout (tiles of
    tile_rows rows; flat u8 of mxg_act_tiled_bytes bytes)."""
    _need(x.is_cuda and x.dtype == torch.bfloat16 and x.dim() == 2 and x.stride(1) == 1,
          "x must be a CUDA bf16 (M, K) tensor with unit inner stride")
    M, K = x.shape
    if codes is None:
        codes = torch.empty(mxg_act_tiled_bytes(KIND_A4W4, M, K, tile_rows), dtype=torch.uint8, device=x.device)
    if sf is None:
        sf = torch.empty(mxg_sf_bytes(M, K, SF_SWIZZLED), dtype=torch.uint8, device=x.device)
    _check("mx_quantize_act_tiled", lib().mx_quantize_act_tiled(
        _ptr(x), M, K, x.stride(0), tile_rows, _ptr(codes), _ptr(sf), _stream(stream)))
    return codes, sf


def fp8_quantize_act_tiled(x: torch.Tensor, tile_rows: int, q=None, scale=None, stream=None):
    """fp8_quantize_act with q in the activation tile layout."""
    _need(x.is_cuda and x.dtype == torch.bfloat16 and x.dim() == 2 and x.stride(1) == 1,
          "x must be a CUDA bf16 (M, K) tensor with unit inner stride")
    M, K = x.shape
    if q is None:
        q = torch.empty(mxg_act_tiled_bytes(KIND_PTPC, M, K, tile_rows), dtype=torch.uint8, device=x.device)
    if scale is None:
        scale = torch.empty(M, dtype=torch.float32, device=x.device)
    _check("fp8_quantize_act_tiled", lib().fp8_quantize_act_tiled(
        _ptr(x), M, K, x.stride(0), tile_rows, _ptr(q), _ptr(scale), _stream(stream)))
    return q, scale


def fp8_quantize_act(x: torch.Tensor, q=None, scale=None, stream=None):
    """Per-row E4M3 quantization: x (M, K) bf16 -> (q (M, K) u8, scale (M,) f32).
    Applied to a weight W (N, K) it gives the per-output-channel conversion."""
    _need(x.is_cuda and x.dtype == torch.bfloat16 and x.dim() == 2 and x.stride(1) == 1,
          "x must be a CUDA bf16 (M, K) tensor with unit inner stride")
    M, K = x.shape
    if q is None:
        q = torch.empty(M, K, dtype=torch.uint8, device=x.device)
    if scale is None:
        scale = torch.empty(M, dtype=torch.float32, device=x.device)
    _check("fp8_quantize_act", lib().fp8_quantize_act(
        _ptr(x), M, K, x.stride(0), _ptr(q), _ptr(scale), _stream(stream)))
    return q, scale


def swiglu_fp8_quantize(gu: torch.Tensor, tile_rows: int = 0, q=None, scale=None, h=None, stream=None):
    """The step between gate_up and down: gu (M, 2I) bf16 [gate | up] ->
    (q, scale) = per-token FP8 of h = bf16(silu(gate) * up); q row-major
    (M, I) or, with tile_rows, flat in the activation tile layout.  Pass
    h (M, I) bf16 to also receive h."""
    _need(gu.is_cuda and gu.dtype == torch.bfloat16 and gu.dim() == 2 and gu.stride(1) == 1
          and gu.shape[1] % 2 == 0, "gu must be a CUDA bf16 (M, 2I) tensor with unit inner stride")
    M, I = gu.shape[0], gu.shape[1] // 2
    if q is None:
        q = (torch.empty(mxg_act_tiled_bytes(KIND_PTPC, M, I, tile_rows), dtype=torch.uint8, device=gu.device)
             if tile_rows else torch.empty(M, I, dtype=torch.uint8, device=gu.device))
    if scale is None:
        scale = torch.empty(M, dtype=torch.float32, device=gu.device)
    if h is not None:
        _need(h.dtype == torch.bfloat16 and h.stride(1) == 1 and tuple(h.shape) == (M, I), "h must be (M, I) bf16")
    _check("swiglu_fp8_quantize", lib().swiglu_fp8_quantize(
        _ptr(gu), M, I, gu.stride(0), int(tile_rows), _ptr(q), _ptr(scale), _ptr(h),
        h.stride(0) if h is not None else 0, _stream(stream)))
    return q, scale


# ---------------------------------------------------------------- GEMMs
def _opts(variant, ctas, ws, dev_status, timeout_ms, debug_stall, weights_static=False,
          trace=None, weights_tiled=False, act_tile_rows=0, splitk_reduce="default",
          cta_pair=False) -> GemmOpts:
    return GemmOpts(variant=VARIANTS[variant], ctas=int(ctas), weights_static=int(weights_static),
                    cta_pair=int(cta_pair),
                    weights_tiled=int(weights_tiled), act_tile_rows=int(act_tile_rows),
                    splitk_reduce=REDUCE[splitk_reduce],
                    trace=0 if trace is None else trace.data_ptr(),
                    workspace=0 if ws is None else ws.data_ptr(),
                    ws_bytes=0 if ws is None else ws.numel() * ws.element_size(),
                    dev_status=0 if dev_status is None else dev_status.data_ptr(),
                    timeout_ms=int(timeout_ms), debug_stall=int(debug_stall))


def _out(out, M, N, out_f32, device):
    if out is None:
        out = torch.empty(M, N, dtype=torch.float32 if out_f32 else torch.bfloat16, device=device)
    _need(out.dtype == (torch.float32 if out_f32 else torch.bfloat16) and out.stride(1) == 1,
          "out dtype/stride mismatch")
    return out


def mx_gemm_a4w4(w_codes: torch.Tensor, w_sf, *, a_codes=None, a_sf=None, x=None,
                 out=None, out_f32: bool = False, variant: str = "auto", ctas: int = 0,
                 ws=None, dev_status=None, timeout_ms: int = 0, debug_stall: int = 0,
                 weights_static: bool = False, trace=None, weights_tiled: int = W_ROWMAJOR,
                 act_tile_rows: int = 0, m: int = 0, n: int = 0, k: int = 0,
                 splitk_reduce: str = "default", cta_pair: bool = False, stream=None):
    """y (M, N) = MXFP4 A4W4 GEMM.  Either (a_codes, a_sf) pre-quantized or
    x (M, K) bf16 (quantized inside the call).  w_sf must be in the 128x4
    tiles; w_codes row-major, or in weight tiles with weights_tiled=W_TILED
    (or True); with weights_tiled=W_PANEL w_codes is flat in 256-row panels
    (scales inside, w_sf None) and n, k give N, K.  With act_tile_rows,
    a_codes is flat in the activation tile layout and m gives M.  cta_pair:
    run a full-tile GEMM of M > 128 on CTA pairs (2-SM MMAs).  dev_status,
    timeout_ms: the bounded-wait controls; debug_stall (test hook): 1 stalls
    the GEMM's epilogue, 2 the activation quantizer of a fused call of more
    than 512 rows, until the limit runs out."""
    if w_codes.dim() == 1:
        _need(n > 0 and k > 0, "flat weight codes need n and k")
        N, K = n, k
    else:
        N, K2 = w_codes.shape
        K = 2 * K2
    fused = a_codes is None
    if fused:
        _need(x is not None and x.dtype == torch.bfloat16 and x.stride(1) == 1, "x (M, K) bf16 needed")
        M = x.shape[0]
        ldx = x.stride(0)
    else:
        M = m if m else a_codes.shape[0]
        ldx = 0
    out = _out(out, M, N, out_f32, w_codes.device)
    if ws is None:
        ws = workspace(mxg_gemm_workspace_bytes(KIND_A4W4, fused, M, N, K, variant, ctas), w_codes.device)
    o = _opts(variant, ctas, ws, dev_status, timeout_ms, debug_stall, weights_static, trace,
              weights_tiled, act_tile_rows, splitk_reduce, cta_pair)
    _check("mx_gemm_a4w4", lib().mx_gemm_a4w4(
        _ptr(a_codes), _ptr(a_sf), _ptr(x), ldx, _ptr(w_codes), _ptr(w_sf), M, N, K,
        _ptr(out), out.stride(0), OUT_F32 if out_f32 else OUT_BF16, ctypes.byref(o), _stream(stream)))
    return out


def fp8_gemm_ptpc(qa: torch.Tensor, sa: torch.Tensor, qw: torch.Tensor, sw: torch.Tensor, *,
                  out=None, out_f32: bool = False, variant: str = "auto", ctas: int = 0,
                  ws=None, dev_status=None, timeout_ms: int = 0, debug_stall: int = 0,
                  weights_static: bool = False, trace=None, weights_tiled: int = W_ROWMAJOR,
                  act_tile_rows: int = 0, k: int = 0, splitk_reduce: str = "default",
                  cta_pair: bool = False, stream=None):
    """y (M, N) = (sum_k qa qw * sa[m]) * sw[n]: FP8 PTPC A8W8 GEMM; qw
    row-major, or in weight tiles with weights_tiled=W_TILED (or True), or
    flat in 256-row panels with weights_tiled=W_PANEL (k gives K); qa
    row-major, or flat in the activation tile layout with act_tile_rows
    (M = len(sa), N = len(sw)).  cta_pair: run a full-tile GEMM of M > 128
    on CTA pairs (2-SM MMAs)."""
    M = sa.numel()
    N = sw.numel()
    if qw.dim() == 1:
        _need(k > 0, "flat weight bytes need k")
        K = k
    else:
        _need(qw.shape[0] == N, "qw rows and len(sw) differ")
        K = qw.shape[1]
    out = _out(out, M, N, out_f32, qa.device)
    if ws is None:
        ws = workspace(mxg_gemm_workspace_bytes(KIND_PTPC, False, M, N, K, variant, ctas), qa.device)
    o = _opts(variant, ctas, ws, dev_status, timeout_ms, debug_stall, weights_static, trace,
              weights_tiled, act_tile_rows, splitk_reduce, cta_pair)
    _check("fp8_gemm_ptpc", lib().fp8_gemm_ptpc(
        _ptr(qa), _ptr(sa), _ptr(qw), _ptr(sw), M, N, K, _ptr(out), out.stride(0),
        OUT_F32 if out_f32 else OUT_BF16, ctypes.byref(o), _stream(stream)))
    return out


def mxg_grouped_workspace_bytes(M_total: int, K: int, E: int) -> int:
    return int(lib().mxg_grouped_workspace_bytes(M_total, K, E))


def mx_gemm_a4w4_grouped(x: torch.Tensor, row_off: torch.Tensor, w_panels: torch.Tensor, *, n: int,
                         out=None, out_f32: bool = False, ws=None, dev_status=None, timeout_ms: int = 0,
                         weights_static: bool = False, trace=None, stream=None):
    """Grouped (MoE) A4W4: x (M_total, K) bf16 with the tokens sorted by
    expert, row_off (E + 1,) int32 on the device (expert e owns rows
    row_off[e] .. row_off[e+1]-1), w_panels flat: E panel sets of
    mxg_weight_bytes(KIND_A4W4, n, K, PANEL) bytes each.  Returns y (M_total, n)."""
    _need(x.is_cuda and x.dtype == torch.bfloat16 and x.dim() == 2 and x.stride(1) == 1,
          "x must be a CUDA bf16 (M, K) tensor with unit inner stride")
    _need(row_off.is_cuda and row_off.dtype == torch.int32 and row_off.dim() == 1 and row_off.is_contiguous(),
          "row_off must be a contiguous CUDA int32 vector")
    M, K = x.shape
    E = row_off.numel() - 1
    out = _out(out, M, n, out_f32, x.device)
    if ws is None:
        ws = workspace(mxg_grouped_workspace_bytes(M, K, E), x.device)
    o = _opts("auto", 0, ws, dev_status, timeout_ms, 0, weights_static, trace)
    _check("mx_gemm_a4w4_grouped", lib().mx_gemm_a4w4_grouped(
        _ptr(x), x.stride(0), _ptr(row_off), E, _ptr(w_panels), M, n, K, _ptr(out), out.stride(0),
        OUT_F32 if out_f32 else OUT_BF16, ctypes.byref(o), _stream(stream)))
    return out


def mxg_mma_peak(kind: int, n: int = 256, iters: int = 20000, stream=None) -> float:
    """TFLOP/s of the GEMMs' MMA instruction shape on operands resident in
    shared memory (all SMs); synchronises the stream."""
    out = ctypes.c_double(0.0)
    _check("mxg_mma_peak", lib().mxg_mma_peak(kind, n, iters, ctypes.byref(out), _stream(stream)))
    return float(out.value)


def mxg_query_status(dev_status: torch.Tensor | None, stream=None) -> int:
    """Synchronise the stream, read and clear the device status word."""
    return int(lib().mxg_query_status(_ptr(dev_status), _stream(stream)))
