/*
 * mxgemm.h -- C ABI of the GB300 (sm_103a) MXFP4 A4W4 / FP8 PTPC A8W8 library.
 *
 * The library implements the quantized linear layers of a mixed-precision
 * speculative-decoding draft model:
 *
 *   - MXFP4 (page "Kimi-K3 DSpark O-Proj-only MXFP4", section "Exact
 *     quantization coverage"): E2M1 element codes, one E8M0 scale per 32
 *     consecutive input-channel values, weight stored (N, K) = (7168, 8192)
 *     with scale (7168, 256); at run time "dynamic MXFP4 activations with
 *     A4W4 dispatch" (the same section).  "OCP MXFP4" names the standard
 *     (page "Kimi-K3-Quark-MXFP4-AttnFP8", section "Model Overview").
 *   - FP8 PTPC (page "Kimi-K3-DSpark-FP8-PTPC", section "Phase 1 FP8 PTPC
 *     Quantization"): E4M3 weights with one FP32 scale per output channel
 *     (shape (out_features, 1)); activations quantized per token at run time,
 *     never calibrated or stored.
 *
 * Conventions for every entry point:
 *   - Linear layout y = x . W^T: x (M, K) and W (N, K) are row-major and
 *     K-contiguous (leading dimensions in ELEMENTS); y (M, N) row-major.
 *   - All tensor pointers are DEVICE pointers owned by the caller; the
 *     library allocates no device memory and keeps no pointer after a call
 *     returns.  Scratch memory, where needed, is the caller's workspace.
 *   - Calls are asynchronous on `stream` (NULL = legacy default stream) and
 *     do not synchronise the host, except mxg_query_status.  Kernels are
 *     launched with programmatic stream serialization: each may begin its
 *     prologue while the kernels before it finish, and touches no memory
 *     they may use before the kernel just before it has completed (which in
 *     turn waited for its own predecessor).  The one exception is the GEMMs'
 *     opts->weights_static.  The weight quantizers (mx_quantize_weight,
 *     fp8_quantize_weight) never let a later kernel start before they end.
 *   - Host-detectable errors (bad shape, alignment, device, workspace) are
 *     returned before anything is launched.  A failed launch returns
 *     MXG_ERR_CUDA.  Device-side waits are bounded; a wait that runs out
 *     ORs MXG_DEV_TIMEOUT into opts->dev_status (if given) and the kernel
 *     returns early, leaving the context usable.  Large inputs (more than
 *     512 rows) of the quantizers stream through shared memory by bulk
 *     copies; a copy wait that runs out leaves the rows not yet quantized
 *     with NaN scales (FP8 s = NaN, MX scale code 0xFF), which make every
 *     product with them NaN.  The quantizer entry points have no status word
 *     (their limit is 1 s); the activation quantizer of a fused mx_gemm_a4w4
 *     call uses opts->dev_status and opts->timeout_ms.
 *   - Requirements: compute capability 10.3 (GB300); K % 128 == 0; M, N >= 1
 *     (N % 128 == 0 for the GEMMs); every pointer 16-byte aligned; every
 *     leading dimension a multiple of 16 bytes.
 *   - Quantization rules (the pages fix the formats, not the rounding; these
 *     are the readings the library and its CPU oracle share):
 *       MX: per block of 32, amax = max|x|; e = clamp(floor(log2 amax) - 2,
 *           -127, 127) (an all-zero block gets e = -127); scale code = e+127;
 *           code = E2M1(x * 2^-e), round to nearest even, saturating, sign
 *           kept (also for -0).  A block holding NaN/Inf gets scale 0xFF and
 *           zero codes.  Two codes per byte, the lower k in the low nibble.
 *       FP8: per row, s = amax / 448 (fp32 division); s = 1 for an all-zero
 *           row; q = E4M3(x / s) (fp32 division, then round to nearest even,
 *           saturating at +-448, sign kept).  A row holding NaN/Inf gets
 *           s = NaN and zero codes.
 */
#ifndef MXGEMM_H
#define MXGEMM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* The same type as cudaStream_t / CUstream. */
typedef struct CUstream_st *mxg_stream_t;

typedef enum {
    MXG_OK = 0,
    MXG_ERR_INVALID_ARG = 1,        /* null pointer, non-positive size, bad enum */
    MXG_ERR_UNSUPPORTED_SHAPE = 2,  /* K % 128 != 0, N % 128 != 0, size too large */
    MXG_ERR_MISALIGNED = 3,         /* pointer or leading dimension not 16-byte aligned */
    MXG_ERR_UNSUPPORTED_DEVICE = 4, /* current device is not compute capability 10.3 */
    MXG_ERR_CUDA = 5,               /* a CUDA runtime/driver call failed */
    MXG_ERR_TIMEOUT = 6,            /* a device-side bounded wait ran out (mxg_query_status) */
    MXG_ERR_WORKSPACE = 7           /* workspace missing or smaller than required */
} mxg_status;

/* Bits a kernel ORs into the optional device status word. */
#define MXG_DEV_TIMEOUT 0x1
#define MXG_DEV_BAD_INDEX 0x2
#define MXG_DEV_SMEM_LAYOUT 0x4 /* a GEMM CTA found its dynamic shared memory less aligned than
                                   its layout needs and did nothing (never seen; reported as
                                   MXG_ERR_CUDA) */

typedef enum {
    MXG_SF_ROWMAJOR = 0, /* (rows, K/32) bytes, row-major: the stored checkpoint layout */
    MXG_SF_SWIZZLED = 1, /* 128x4 tiles of 512 bytes (see mxg_sf_bytes); the GEMM operand layout */
    MXG_TILED = 2,       /* scales as MXG_SF_SWIZZLED, and the codes in the GEMM's weight tile
                            layout (see MXG_TILE_BYTES); needs rows % 128 == 0 and, for MXFP4,
                            K % 256 == 0 */
    MXG_PANEL = 3        /* weights only: the codes in 256-row panels with the MXFP4 scales
                            inside them (see MXG_PANEL_ROWS); K % 256 == 0 for MXFP4 */
} mxg_sf_layout;

/* Weight tile layout (MXG_TILED), for MXFP4 codes and for FP8 E4M3 bytes alike:
 * a row is cut into 128-byte chunks (256 FP4 or 128 FP8 values, KC = row bytes
 * / 128 chunks); the 128 rows x 128 bytes of row block rb and chunk kc form one
 * 16 KiB tile at byte ((rb * KC) + kc) * 16384; inside it, the 16-byte unit j
 * (0..7) of row r (0..127) sits at r * 128 + ((j ^ (r % 8)) * 16).  That is the
 * shared-memory image the tensor cores read (K-major, 128-byte swizzle), so a
 * GEMM stage fetches a weight tile with one contiguous bulk copy. */
#define MXG_TILE_BYTES 16384

/* Weight panel layout (MXG_PANEL): the rows are grouped in panels of 256
 * (the last panel padded with zero codes).  Panel p and chunk kc form one
 * block at byte (p * KC + kc) * B, B = 34816 for MXFP4 and 32768 for FP8:
 * first the two 128-row halves of the panel, each a 16 KiB tile as in
 * MXG_TILED (half h at h * 16384, row r of the weight being row r % 128 of
 * half (r / 128) % 2 of panel r / 256); then, MXFP4 only, the scales of the
 * chunk's 8 groups: half h at 32768 + h * 1024, the 2 x 512-byte 128x4 tiles
 * of MXG_SF_SWIZZLED for groups 8kc..8kc+3 and 8kc+4..8kc+7 (tile
 * offsets as in mxg_sf_bytes, with r % 128).  A full-tile GEMM stage (256
 * weight rows, one chunk) then fetches its whole weight operand, codes and
 * scales, with one bulk copy.  Bytes: mxg_weight_bytes. */
#define MXG_PANEL_ROWS 256

typedef enum {
    MXG_OUT_BF16 = 0, /* y rounded to bf16 (round to nearest even) */
    MXG_OUT_F32 = 1   /* y in fp32 before the bf16 cast (test / parity mode) */
} mxg_out_dtype;

typedef enum {
    MXG_VARIANT_AUTO = 0,   /* the dispatcher chooses from (M, N, K, SM count) */
    MXG_VARIANT_FULL = 1,   /* one CTA owns a whole output tile and all of K */
    MXG_VARIANT_SPLITK = 2  /* operands swapped (weights fill the 128-row MMA side),
                               K split across CTAs (stream-K), fixed-order reduction */
} mxg_variant;

typedef struct {
    int variant;          /* mxg_variant */
    int ctas;             /* SPLITK: number of CTAs to spread the K-blocks over (stream-K);
                             more than the SM count = the SM count (one persistent CTA per
                             SM).  0 = the dispatcher's choice: the SM count, or one CTA per
                             whole tile (no partial sums, no reduce kernel) when the tiles
                             fit on the SMs and a tile's K-stages are at most a stream-K
                             CTA's share plus 7 (the measured cost of the reduce kernel) */
    void *workspace;      /* device scratch of >= mxg_gemm_workspace_bytes() bytes,
                             256-byte aligned: the fused path's quantized activations, then
                             the split-K partial tiles.  Its contents on entry do not
                             matter.  Calls that overlap on the GPU need separate
                             workspaces.  NULL only when the call needs none. */
    size_t ws_bytes;      /* size of workspace */
    int *dev_status;      /* optional device int; kernels OR MXG_DEV_* bits into it */
    uint32_t timeout_ms;  /* limit of every device-side wait; 0 = 1000 ms */
    int debug_stall;      /* test hook: 1 makes the epilogue wait on a barrier nothing
                             arrives at, so the timeout path runs (no fault, no hang);
                             2 does the same in the activation quantizer of a fused
                             mx_gemm_a4w4 call of more than 512 rows, which then
                             leaves NaN scales (0xFF), so the GEMM writes NaN rows */
    int weights_static;   /* 1: no kernel that may still be running when the GEMM starts
                             writes the weight operands (w_codes/w_sf or qw/sw), so the
                             GEMM may stream them in before the kernels ahead of it on
                             `stream` have finished (programmatic dependent launch).
                             Weights written by mx_quantize_weight / fp8_quantize_weight,
                             by a kernel without programmatic launch, or before a
                             synchronisation qualify; weights written by this library's
                             activation quantizers, GEMMs or reduce do not. */
    int weights_tiled;    /* 0: w_codes (A4W4) / qw (PTPC) are row-major; 1: in the
                             MXG_TILED weight tile layout; 2: in the MXG_PANEL layout (A4W4:
                             w_sf is then unused and may be NULL) */
    int act_tile_rows;    /* 0: a_codes (A4W4) / qa (PTPC) are row-major; else they are in
                             the activation tile layout with tiles of this many rows, as
                             written by mx_quantize_act_tiled / fp8_quantize_act_tiled; it
                             must equal the plan's MMA-N tile (mxg_plan_gemm().bn) for the
                             SPLITK variant and 128 for the FULL variant.  (The fused A4W4
                             path picks its own layout and ignores this field.) */
    void *trace;          /* optional device buffer of ctas x 40 uint64, zero-filled: each
                             CTA records SM clock64 stamps of its timeline (entry, setup,
                             first/last load, first stage ready, last MMA commit, epilogue
                             items, split-K partial stored, exit; slot 15 = items; slots
                             16/17 = global timer ns at entry/exit; slot 18 = the
                             producer's dependency wait returned, slot 20 = the same in
                             global timer ns).  Slots 22
                             and 23 of CTA 0's row: the split-K reduce kernel of the same
                             call, ~(first entry ns) and last exit ns.  Slot 21: the SM.
                             A4W4, slots 24+k / 32+k: the CTA's k-th pipeline stage
                             (k < 8) landed in shared memory / its scales are in TMEM.
                             NULL = off. */
    int splitk_reduce;    /* MXG_REDUCE_DEFAULT or MXG_REDUCE_KERNEL (the same): SPLITK
                             partial tiles are summed, in slot order, by a reduce kernel
                             launched right after the GEMM.  Any other value is
                             MXG_ERR_INVALID_ARG.  On the fused A4W4 path (x given) the
                             call launches the activation quantizer, the GEMM and the
                             reduce kernel, chained by programmatic dependent launch. */
    int cta_pair;         /* FULL variant, M > 128: 1 = run the tiles on clusters of two CTAs
                             issuing 2-SM MMAs (tcgen05 cta_group::2) over 256-token x
                             256-channel tiles, each CTA holding 128 token rows and one
                             128-row half of the weight tile (a third fewer operand bytes
                             per flop); 0 (default) = one CTA per 128 x 256 tile, which
                             measured faster on this part (the MMA issue loop, not operand
                             bytes, bounds both).  Not for mx_gemm_a4w4_grouped (must be 0). */
} mxg_gemm_opts;

enum {
    MXG_REDUCE_DEFAULT = 0,
    MXG_REDUCE_KERNEL = 1
};

typedef struct {
    int variant;       /* MXG_VARIANT_FULL or MXG_VARIANT_SPLITK */
    int bm, bn;        /* output tile: bm rows of the MMA-A operand (tokens for FULL,
                          weight rows for SPLITK), bn of the MMA-B operand */
    int ctas;          /* grid size */
    int tiles;         /* output tiles */
    int kblocks;       /* pipeline stages along K per tile: 128-byte K columns (256 K
                          for A4W4, 128 K for PTPC), one per stage for FULL, two for
                          SPLITK */
    int seg_max;       /* SPLITK: most CTAs contributing to one tile */
    size_t ws_bytes;   /* workspace this plan needs (partial tiles) */
    int cta_pair;      /* FULL: 1 = clusters of two CTAs issuing 2-SM MMAs (tcgen05
                          cta_group::2) over 256-token x 256-channel tiles, each CTA holding
                          128 token rows and one 128-row half of the weight tile (requested
                          with mxg_gemm_opts.cta_pair and M > 128); 0 = one CTA per
                          128 x 256 tile */
} mxg_plan;

/* Bytes of a scale-factor array for `rows` rows of K elements (K/32 groups).
 * ROWMAJOR: rows * K/32.  SWIZZLED: ceil(rows/128)*128 * K/32: the scale of
 * (row r, group g) sits at ((r/128)*(G/4) + g/4)*512 + (r%32)*16 +
 * ((r%128)/32)*4 + g%4 with G = K/32; padding rows hold 0. */
size_t mxg_sf_bytes(int rows, int K, mxg_sf_layout layout);

/* Bytes of a quantized weight's codes (kind 0: MXFP4, K/2 bytes a row; kind 1:
 * FP8, K bytes a row) in `layout`: N * row bytes, or for MXG_PANEL
 * ceil(N/256) * (row bytes / 128) * (34816 | 32768) (scales included);
 * 0 for an invalid argument. */
size_t mxg_weight_bytes(int kind, int N, int K, mxg_sf_layout layout);

/* Dispatcher, pure host logic (no GPU needed): the variant, tile and grid a
 * GEMM of kind 0 (A4W4) or 1 (PTPC) at (M, N, K) would use on a device with
 * `sm_count` SMs under `opts` (nullable), and the workspace it needs. */
mxg_status mxg_plan_gemm(int kind, int M, int N, int K, int sm_count,
                         const mxg_gemm_opts *opts, mxg_plan *plan);

/* Workspace bytes mx_gemm_a4w4 (kind 0, fused == 0), mx_gemm_a4w4 with bf16
 * activations (kind 0, fused == 1) or fp8_gemm_ptpc (kind 1) needs on the
 * current device with `opts` (nullable); 0 if none. */
size_t mxg_gemm_workspace_bytes(int kind, int fused, int M, int N, int K,
                                const mxg_gemm_opts *opts);

/* Offline MXFP4 weight conversion ("Exact quantization coverage": E2M1 codes,
 * E8M0 scale per 32 consecutive input channels).
 *   w_bf16: (N, K) bf16, leading dimension ldw elements.
 *   codes:  N * K/2 bytes, two codes per byte, lower k in the low nibble:
 *           row-major (N, K/2) for ROWMAJOR / SWIZZLED, weight tiles for TILED,
 *           mxg_weight_bytes(0, N, K, MXG_PANEL) bytes of panels for PANEL.
 *   sf:     mxg_sf_bytes(N, K, layout) bytes, ROWMAJOR (the stored (N, K/32)
 *           checkpoint layout) or the 128x4 tiles (SWIZZLED, TILED); unused
 *           (may be NULL) for PANEL, whose scales sit inside the panels. */
mxg_status mx_quantize_weight(const void *w_bf16, int N, int K, int ldw,
                              uint8_t *codes, uint8_t *sf, mxg_sf_layout layout,
                              mxg_stream_t stream);

/* Dynamic MXFP4 activation quantization ("dynamic MXFP4 activations with
 * A4W4 dispatch"): per row of x (M, K) bf16, per block of 32.
 *   codes: (M, K/2) bytes.  sf: mxg_sf_bytes(M, K, MXG_SF_SWIZZLED) bytes
 *   (padding rows are written as 0). */
mxg_status mx_quantize_act(const void *x_bf16, int M, int K, int ldx,
                           uint8_t *codes, uint8_t *sf, mxg_stream_t stream);

/* Block-scaled A4W4 GEMM ("A4W4 dispatch"): y[m][n] = sum_g 2^(ea[m,g]-127) *
 * 2^(ew[n,g]-127) * sum_{k in g} v(a[m,k]) v(w[n,k]), fp32 accumulation,
 * then bf16 (or fp32) output.
 *   a_codes (M, K/2) + a_sf (swizzled): pre-quantized activations, OR
 *   a_codes == NULL and x_bf16 (M, K) with leading dimension ldx: the
 *   activations are quantized inside the call (codes and scales identical to
 *   mx_quantize_act) into the workspace.
 *   w_codes (N, K/2), w_sf (swizzled): the weight, row-major codes, or the
 *   codes in the layout opts->weights_tiled names (MXG_TILED tiles, or
 *   MXG_PANEL panels whose scales sit inside them: w_sf is then unused).
 *   a_codes in the activation tile layout when opts->act_tile_rows != 0.
 *   y: (M, N) with leading dimension ldy elements, bf16 or fp32. */
mxg_status mx_gemm_a4w4(const uint8_t *a_codes, const uint8_t *a_sf,
                        const void *x_bf16, int ldx,
                        const uint8_t *w_codes, const uint8_t *w_sf,
                        int M, int N, int K, void *y, int ldy, mxg_out_dtype out_dtype,
                        const mxg_gemm_opts *opts, mxg_stream_t stream);

/* Dynamic per-token FP8 quantization (and, applied to W rows, the
 * per-output-channel weight conversion of "Phase 1 FP8 PTPC Quantization").
 *   x_bf16 (M, K), leading dimension ldx.  q: (M, K) E4M3 bytes.
 *   scale: M floats (the (out_features, 1) scale when x is a weight). */
mxg_status fp8_quantize_act(const void *x_bf16, int M, int K, int ldx,
                            uint8_t *q, float *scale, mxg_stream_t stream);

/* Per-output-channel FP8 weight conversion ("Phase 1 FP8 PTPC Quantization":
 * E4M3 weight, FP32 scale of shape (out_features, 1)); the same arithmetic as
 * fp8_quantize_act applied to the rows of W.
 *   w_bf16 (N, K), leading dimension ldw.  q: N * K bytes, row-major (N, K)
 *   for MXG_SF_ROWMAJOR, weight tiles for MXG_TILED (N % 128 == 0), or
 *   mxg_weight_bytes(1, N, K, MXG_PANEL) bytes of panels for MXG_PANEL.
 *   scale: N floats. */
mxg_status fp8_quantize_weight(const void *w_bf16, int N, int K, int ldw,
                               uint8_t *q, float *scale, mxg_sf_layout layout,
                               mxg_stream_t stream);

/* Activation tile layout: the weight tile layout (MXG_TILE_BYTES) with tiles
 * of T = tile_rows rows instead of 128 (T in {16, 32, 64, 128, 256}): tile
 * (r / T, chunk kc) of T rows x 128 bytes at byte ((r/T) * KC + kc) * T * 128,
 * the 16-byte unit j of row r at (r % T) * 128 + ((j ^ (r % 8)) * 16).  The
 * GEMM fetches a token tile with one bulk copy.  Rows past M in the last tile
 * are left unwritten (they only feed output columns past M, which are not
 * stored).  Bytes: mxg_act_tiled_bytes. */
size_t mxg_act_tiled_bytes(int kind, int M, int K, int tile_rows);

/* mx_quantize_act with the codes in the activation tile layout (K % 256 == 0);
 * the scales as mx_quantize_act (128x4 tiles, padding rows 0). */
mxg_status mx_quantize_act_tiled(const void *x_bf16, int M, int K, int ldx, int tile_rows,
                                 uint8_t *codes, uint8_t *sf, mxg_stream_t stream);

/* fp8_quantize_act with q in the activation tile layout. */
mxg_status fp8_quantize_act_tiled(const void *x_bf16, int M, int K, int ldx, int tile_rows,
                                  uint8_t *q, float *scale, mxg_stream_t stream);

/* The step between the packed gate_up projection and the down projection of
 * the FP8 MLP ("Phase 1 FP8 PTPC Quantization": gate_proj and up_proj are
 * packed into one gate_up_proj), fused with the down projection's dynamic
 * per-token FP8 quantization.  The pages do not name the activation; the
 * library takes SwiGLU:
 *   h[m][j] = bf16(silu(g) * u),  g = gu[m][j], u = gu[m][I + j],
 *   silu(g) * u = (g / (1 + e^-g)) * u in binary32, one IEEE operation at a
 *   time, e^t by the Cody-Waite method (t = n ln2 + r, Taylor series of e^r
 *   through r^7/7!), so the result is the same on any IEEE machine;
 * then q, scale = fp8_quantize_act(h) (per row: s = amax/448, q = E4M3(h/s)).
 *   gu_bf16: (M, 2I) bf16, a row [gate (I) | up (I)], leading dimension ldgu
 *            (>= 2I elements).  I % 128 == 0, I <= 102400.
 *   q:       E4M3 codes of h, row-major (M, I) for tile_rows == 0, else in
 *            the activation tile layout with tiles of tile_rows rows (as
 *            fp8_quantize_act_tiled writes; what fp8_gemm_ptpc reads with
 *            opts->act_tile_rows = tile_rows).  scale: M floats.
 *   h_bf16:  optional (NULL = not written) (M, I) bf16 output of h itself,
 *            leading dimension ldh. */
mxg_status swiglu_fp8_quantize(const void *gu_bf16, int M, int I, int ldgu, int tile_rows,
                               uint8_t *q, float *scale, void *h_bf16, int ldh,
                               mxg_stream_t stream);

/* FP8 PTPC A8W8 GEMM: y[m][n] = (acc[m][n] * sa[m]) * sw[n] with
 * acc = sum_k v(qa[m,k]) v(qw[n,k]) accumulated in fp32.
 *   qa (M, K), sa (M); qw (N, K), sw (N); y (M, N), leading dimension ldy.
 *   qw row-major, or in the layout opts->weights_tiled names (MXG_TILED /
 *   MXG_PANEL); qa in the activation tile layout when opts->act_tile_rows
 *   != 0. */
mxg_status fp8_gemm_ptpc(const uint8_t *qa, const float *sa,
                         const uint8_t *qw, const float *sw,
                         int M, int N, int K, void *y, int ldy, mxg_out_dtype out_dtype,
                         const mxg_gemm_opts *opts, mxg_stream_t stream);

/* Grouped (MoE) A4W4 GEMM for the experts of a mixture-of-experts layer
 * (page "Kimi-K3-Quark-MXFP4-AttnFP8", section "Model Overview": the experts
 * are OCP MXFP4): the token rows arrive grouped by expert, and each group goes
 * through its own expert's MXFP4 weight,
 *   y[row_off[e] + i][n] = sum_k x_q[row_off[e] + i][k] * W_e_q[n][k]
 * for i < row_off[e+1] - row_off[e], with x quantized inside the call (dynamic
 * MXFP4, codes and scales as mx_quantize_act) and fp32 accumulation.  The
 * routing and the token permutation that produce the grouping are not part of
 * this call.
 *   x_bf16:   (M_total, K) bf16, the tokens sorted by expert, leading dimension
 *             ldx elements.
 *   row_off:  DEVICE array of E + 1 ints: expert e owns rows row_off[e] ..
 *             row_off[e+1] - 1; row_off[0] = 0, row_off[E] = M_total, non-
 *             decreasing (empty groups allowed).  1 <= E <= 1024.
 *   w_panels: E weight panel sets (MXG_PANEL, as mx_quantize_weight writes),
 *             expert e at byte e * mxg_weight_bytes(0, N, K, MXG_PANEL).
 *   y:        (M_total, N) bf16 or fp32, leading dimension ldy, rows in x's
 *             order.
 *   opts:     required; workspace of >= mxg_grouped_workspace_bytes(M_total, K,
 *             E) bytes (256-byte aligned; its contents on entry do not matter);
 *             variant AUTO or FULL (the full-tile kernel: 128-token x 256-
 *             channel tiles, each expert's tokens starting a new tile);
 *             dev_status, timeout_ms, weights_static and trace as for
 *             mx_gemm_a4w4.
 *   K % 256 == 0, N % 128 == 0.  M_total == 0 launches nothing (x and y may
 *   then be NULL). */
size_t mxg_grouped_workspace_bytes(int M_total, int K, int E);
mxg_status mx_gemm_a4w4_grouped(const void *x_bf16, int ldx, const int *row_off, int E,
                                const uint8_t *w_panels, int M_total, int N, int K,
                                void *y, int ldy, mxg_out_dtype out_dtype,
                                const mxg_gemm_opts *opts, mxg_stream_t stream);

/* Size of the library-owned scratch array used by mx_gemm_a4w4_noalloc. */
#define MXG_NOALLOC_SCRATCH_BYTES (16u << 20)

/* mx_gemm_a4w4 for callers that cannot allocate device memory.  The pages
 * have no counterpart: this is a library convenience, not part of the method.
 * Some callers own every device byte themselves and hand a kernel only its
 * inputs and outputs -- for example the custom-op or plugin interface of an
 * inference engine that plans all memory up front, or a serving loop that
 * must not allocate on its hot path because an allocation can stall on a
 * device-wide synchronisation or fail when memory is fragmented.  This entry
 * point takes the same operands as mx_gemm_a4w4 (default dispatch; weights in
 * the layout weights_tiled names, as in mxg_gemm_opts) and no workspace: its scratch
 * is a file-scope device array of MXG_NOALLOC_SCRATCH_BYTES (16 MiB) inside
 * the library, which every GPU that loads the library keeps until the
 * process exits.  It calls no cudaMalloc/cudaFree or any allocating routine.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture.
 *   - Shapes whose scratch would exceed the array (see
 *     mxg_gemm_workspace_bytes) return MXG_ERR_WORKSPACE before any launch.
 *   - Every byte of the array a call reads, that call has written first, so
 *     nothing needs clearing between calls.  All calls share the one array,
 *     which keeps the last call's contents: calls that overlap on the GPU
 *     (other streams, other threads) race on it and must be serialised by
 *     the caller.
 *   - Every operand is checked before the scratch is touched: a call that
 *     returns an error has written nothing.
 *   - It has no device status word: a bounded device wait that runs out
 *     ends the kernel early (y then partly written) without being reported.
 *     Callers that need that report use mx_gemm_a4w4 with opts->dev_status. */
mxg_status mx_gemm_a4w4_noalloc(const uint8_t *a_codes, const uint8_t *a_sf,
                                const void *x_bf16, int ldx,
                                const uint8_t *w_codes, const uint8_t *w_sf,
                                int M, int N, int K, void *y, int ldy, mxg_out_dtype out_dtype,
                                int weights_tiled, mxg_stream_t stream);

/* Synchronises `stream`, reads the device status word, clears it, and maps
 * it: MXG_OK, MXG_ERR_TIMEOUT (MXG_DEV_TIMEOUT set) or MXG_ERR_CUDA. */
mxg_status mxg_query_status(int *dev_status, mxg_stream_t stream);

/* Measurement utility (no counterpart on the pages): the rate of this
 * library's tcgen05 MMA instruction shape with the operands already in shared
 * memory -- the ceiling the GEMMs' main loops run against.  One CTA per SM,
 * one thread issuing `iters` x 4 MMAs of M = 128, N = n (128 or 256), K = 64
 * block-scaled E2M1 (kind 0, scales resident in TMEM) or K = 32 E4M3 (kind 1)
 * into one TMEM accumulator; timed with CUDA events on `stream`, which it
 * synchronises.  *tflops = dense TFLOP/s over all SMs.  It allocates (and
 * frees) one int of device memory. */
mxg_status mxg_mma_peak(int kind, int n, int iters, double *tflops, mxg_stream_t stream);

/* Human-readable name of a status code (static string). */
const char *mxg_status_string(mxg_status s);

#ifdef __cplusplus
}
#endif

#endif /* MXGEMM_H */
