/*
 * moe.h -- C ABI of a single-GPU mixture-of-experts layer for NVIDIA GB300
 * (sm_103a): router top-k, device-side schedule, dispatch gather, grouped
 * expert GEMMs (BF16 or OCP MXFP8) with fused SwiGLU and quantisation,
 * deterministic combine, an optional BF16 shared expert, and the backward
 * pass.
 *
 * The method is the one described by the "Mixture-of-Kittens" pages (Cursor's
 * MoE training megakernel): token routing, a device-side schedule kernel with
 * no CPU synchronisation, dispatch, expert grouped GEMMs with SwiGLU and
 * activation quantisation fused in, and a bitwise-deterministic combine
 * ("Mixture-of-Kittens" wiki page, TL;DR, flowchart and Key claims).  The
 * pages' inter-GPU dispatch/combine become intra-GPU gathers here.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - All pointers are DEVICE pointers unless stated otherwise; the caller owns
 *   every buffer.  The library allocates nothing and keeps no per-call state.
 * - Every tensor is row-major and contiguous.  bf16 = IEEE bfloat16 bits.
 *   Pointers must be 16-byte aligned (MOE_ERR_ALIGN otherwise).
 * - Every call is asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *   default stream): no host synchronisation, no device-to-host copy.  Only
 *   moe_get_status synchronises.
 * - Return value: MOE_OK (0), or a negative moe_status for errors detected on
 *   the host before anything is launched.  Errors detected on the device
 *   (a bounded wait that ran out) are recorded in the status word inside the
 *   workspace and read with moe_get_status.
 * - Results are bitwise reproducible: the same inputs give the same bits on
 *   every call (fixed floating-point operation order, no atomics on floats).
 *
 * MXFP8 format (OCP Microscaling v1.0, as the layer's MXFP8 configurations
 * state): codes are E4M3 bytes; every 32 consecutive elements along the
 * reduction axis K share one E8M0 scale byte (2**(byte-127)); the shared
 * exponent is floor(log2(amax)) - 8, clamped to [-127, 127] (an all-zero
 * block gets byte 0); codes are round-to-nearest-even and saturate to +-448.
 *
 * MXFP8 scale layouts.  A matrix with `rows` rows and reduction length K has
 * rows*K/32 scale bytes.
 *   Canonical (every scale this ABI takes from or returns to the caller):
 *     [rows, K/32] row-major, the scale of (row r, block b = column/32) at
 *     byte r*(K/32) + b.  Batched matrices stack along rows.
 *   Prepared (the expert GEMMs' operand layout; internal): the same bytes in
 *     the order the tensor cores' scale-factor copy reads them, made from
 *     canonical scales by moe_prepare_scales and turned back by
 *     moe_canonical_scales (rows and K multiples of 128).  moe_weights'
 *     *_scale fields and the scale buffers inside the workspace use it.  For
 *     reference, byte ((r/128)*(K/128) + b/4)*512 + (r%32)*16 + ((r%128)/32)*4
 *     + b%4 holds the scale of (r, b): 512-byte atoms of 128 rows x 4 blocks.
 */
#ifndef MOE_H
#define MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *moe_stream_t; /* same type as cudaStream_t */

typedef enum { MOE_BF16 = 0, MOE_MXFP8 = 1, MOE_NVFP4 = 2 } moe_dtype;

typedef enum {
  MOE_OK = 0,
  MOE_ERR_ARG = -1,     /* NULL pointer, non-positive size, k > E, unknown name */
  MOE_ERR_SHAPE = -2,   /* shape outside what the kernels tile (see moe_config) */
  MOE_ERR_ALIGN = -3,   /* a pointer is not 16-byte aligned */
  MOE_ERR_CUDA = -4,    /* a CUDA runtime / driver call or a launch failed */
  MOE_ERR_DEVICE = -5,  /* current device is not sm_103 / sm_100 family */
  MOE_ERR_TIMEOUT = -6, /* device side: a bounded wait inside a kernel ran out */
  MOE_ERR_BOUNDS = -7   /* device side, debug builds only (compiled with -DMOE_DEBUG): an index
                           read from a buffer fell outside its range; the access was skipped */
} moe_status;

/* moe_config.flags bits */
#define MOE_FLAG_BACKWARD 1 /* size the workspace for moe_backward as well */
/* Test hook for the device-side failure path: in moe_forward the gate/up
 * GEMM's load warp issues nothing (with a ring: the gather CTAs publish no
 * tile), so the waits for its data run out (limit 50 ms instead of 4 s); the
 * kernels drain and return, moe_get_status then reports MOE_ERR_TIMEOUT, and
 * the outputs of that call are undefined.  The CUDA context stays usable. */
#define MOE_FLAG_DEBUG_STARVE 2
/* Test hook for the fused quantisation points (MXFP8 experts; ignored with
 * BF16 experts): moe_forward also stores the fp32 SwiGLU output h -- the
 * values the gate/up GEMM's epilogue quantises -- in the workspace buffer
 * "h_dump" [padded rows, m] fp32, and moe_backward stores the bf16 dG|dU
 * values the SwiGLU-backward epilogue quantises in "dGU_dump" [padded rows,
 * 2m] bf16 (moe_buffer_info gives their offsets).  Quantising those dumps
 * with the format's definition must reproduce the codes and scales the
 * kernels wrote, byte for byte.  Nothing else changes.  Not available with a
 * dispatch ring (ring_rows > 0: MOE_ERR_ARG). */
#define MOE_FLAG_DEBUG_DUMP 4

/*
 * Layer shape.  T tokens, hidden d, expert intermediate m, E experts, top-k k.
 * Supported: 1 <= k <= min(E, 16), E <= 1024, d % 256 == 0, m % 128 == 0,
 * m_shared % 128 == 0 (0 = no shared expert), T*k < 2^31 - 127*E.  dtype is
 * the routed experts' arithmetic; the shared expert is always BF16.
 * MOE_NVFP4 (the NVFP4 variant of the expert GEMMs; the pages say the method
 * has none -- "Mixture-of-Kittens" wiki page, Key claims, MXFP8 bullet -- so
 * the format is NVIDIA's published NVFP4): packed E2M1 codes with an E4M3
 * scale per 16 along K and an fp32 second-level scale per tensor (2688 /
 * amax): x's over all T tokens, each expert matrix's own, and 1 for h.
 * Forward only (inference: MOE_FLAG_BACKWARD, a ring or a `saved` buffer give
 * MOE_ERR_ARG) and m % 256 == 0.  flags:
 * any of MOE_FLAG_BACKWARD, MOE_FLAG_DEBUG_STARVE and MOE_FLAG_DEBUG_DUMP, or 0
 * (moe_backward needs a workspace sized with MOE_FLAG_BACKWARD).
 *
 * Dispatch ring (MXFP8 only; "Mixture-of-Kittens" wiki page, flowchart, and
 * daily-ai-frontier summary, TL;DR: a fixed-size token ring between the
 * dispatch and the expert GEMMs, and an SM split between data movement and
 * GEMM work handing off through device counters):
 *   ring_rows  = 0: the dispatch writes every routed row to the workspace
 *                (one row per routed (token, expert) pair, padded per expert);
 *              > 0: a multiple of 128.  The forward's dispatch and gate/up
 *                GEMM run as one persistent launch: `gather_sms` SMs gather
 *                and quantise 128-row tiles of expert-sorted rows into a ring
 *                of ring_rows rows in the workspace, the other SMs run the
 *                GEMM on the ring, and each slot is refilled once every GEMM
 *                tile has loaded it.  Experts with more rows than the ring
 *                pass through it in pieces.  Results are bitwise identical to
 *                ring_rows = 0 for every ring size and SM split.
 *   gather_sms = gather SMs of the ring launch (0 = 8; at most 64).
 *   The ring needs d <= 8192 (MOE_ERR_SHAPE otherwise).
 *
 * Load-balancing term (aux_alpha > 0; the pages define none, so this is the
 * Switch-Transformer auxiliary loss taken over the k routed slots):
 *   L = aux_alpha * E * sum_e f_e * P_e,  f_e = counts_e / (T k),
 *   P_e = (1/T) sum_t softmax(logits_t)_e over all E experts.
 * moe_forward computes it after the schedule (fixed-order sums, bitwise
 * reproducible) into the workspace buffer "aux" = [L, P[E], f[E]] fp32
 * (moe_buffer_info); a training forward also keeps dL/dlogits =
 * aux_alpha E / T * p (f - sum_e f_e p_e), which moe_backward adds to
 * dlogits (the loss enters the objective with weight 1; f is piecewise
 * constant, so no gradient flows through the counts).
 */
typedef struct {
  int32_t T, d, m, E, k;
  int32_t m_shared;
  int32_t dtype; /* moe_dtype */
  int32_t flags;
  int32_t ring_rows;
  int32_t gather_sms;
  float aux_alpha; /* 0 = no load-balancing term */
} moe_config;

/*
 * Expert weights.  BF16 path: `gu` [E, 2m, d] bf16 (rows 0..m-1 of each
 * expert are the gate projection, m..2m-1 the up projection), `dn` [E, d, m]
 * bf16; the *_scale pointers are unused.
 * MXFP8 path: `gu` = E4M3 codes [E*2m, d] with prepared scales `gu_scale`
 * (rows E*2m, K d); `dn` = codes [E*d, m], `dn_scale` (rows E*d, K m) --
 * the codes from moe_quantize_weights(blocks_along_rows = 0) (or
 * moe_quantize_mx(transpose = 0)) of the bf16 masters, the scales that call's
 * canonical scales passed through moe_prepare_scales (an MXFP8 checkpoint's
 * codes and canonical scales can be used the same way).
 * Backward operands (NULL for a forward-only layer):
 *   BF16:  gu_t = [E, d, 2m] bf16 = per-expert transpose of gu,
 *          dn_t = [E, m, d] bf16 = per-expert transpose of dn
 *          (moe_transpose_bf16);
 *   MXFP8: gu_t = codes [E*d, 2m] + prepared gu_t_scale, dn_t = codes
 *          [E*m, d] + prepared dn_t_scale (moe_quantize_weights(
 *          blocks_along_rows = 1) of the masters, then moe_prepare_scales;
 *          moe_quantize_mx_both writes both orientations at once).
 * NVFP4 path: `gu` = packed E2M1 codes [E*2m, d/2] (element 2i in the low
 * nibble of byte i) with prepared E4M3 scales `gu_scale` (rows E*2m, 16-blocks
 * along d), `dn` = [E*d, m/2] with `dn_scale`, and the experts' second-level
 * scales gu_gscale [E], dn_gscale [E] fp32 -- all from moe_prepare_weights.
 * Shared expert (BF16 always; NULL when m_shared == 0): s_gu [2m_s, d],
 * s_dn [d, m_s]; for backward also s_gu_t [d, 2m_s], s_dn_t [m_s, d].
 */
typedef struct {
  const void *gu, *gu_scale;
  const void *dn, *dn_scale;
  const void *gu_t, *gu_t_scale;
  const void *dn_t, *dn_t_scale;
  const void *s_gu, *s_dn;
  const void *s_gu_t, *s_dn_t;
  const float *gu_gscale, *dn_gscale; /* NVFP4 only: second-level scales [E] */
} moe_weights;

/* Bytes of scratch (`ws`) that moe_route / moe_forward / moe_backward need
 * for this config (one buffer serves all three; 0 on invalid config). */
size_t moe_workspace_bytes(const moe_config *cfg);

/* Bytes of the activations a training forward saves for the backward
 * (`saved`; 0 on invalid config). */
size_t moe_saved_bytes(const moe_config *cfg);

/* Byte offset and size of a named sub-buffer of `saved` (which = 0) or of the
 * workspace (which = 1), for inspection by tests and tools.  Names include
 * "idx", "w", "counts", "offsets", "perm", "inv", "poff", "o", "GU", "s_GU",
 * "s_h", with BF16 experts "h" and with MXFP8 experts "xT", "xT_sf", "hT",
 * "hT_sf" (saved: column-blocked codes of the wgrad operands); "xs",
 * "xs_sf", "hq", "hq_sf", "s_out", "dX", "g" and, with MXFP8 experts,
 * "dOq", "dOq_sf", "dOT", "dOT_sf", "dGUq", "dGUq_sf", "dGUT", "dGUT_sf"
 * and, with MOE_FLAG_DEBUG_DUMP, "h_dump" and "dGU_dump"
 * (workspace; "dO" and "dGU" exist only with BF16 experts, whose backward
 * materialises them in bf16).  Row-indexed buffers use padded rows (see
 * moe_forward).  Returns MOE_OK or MOE_ERR_ARG (unknown name / buffer absent
 * for this config). */
int moe_buffer_info(const moe_config *cfg, int which, const char *name, size_t *offset,
                    size_t *bytes);

/* Number of padded expert-sorted rows the buffers are sized for:
 * roundup(T*k + 127*E, 128). */
int64_t moe_padded_rows(const moe_config *cfg);

/*
 * S0: MXFP8 weight quantisation ("Mixture-of-Kittens" wiki page, Key claims,
 * MXFP8 bullet: MXFP8 is the default expert format).
 * src: [batch, rows, cols] bf16.
 *   transpose = 0: codes [batch*rows, cols], blocks of 32 along cols;
 *                  canonical scales [batch*rows, cols/32].
 *   transpose = 1: codes [batch*cols, rows] = per-batch transpose, blocks of
 *                  32 along the original rows; canonical scales
 *                  [batch*cols, rows/32].
 * rows and cols must be multiples of 128.  Inputs must be finite.
 */
int moe_quantize_mx(const void *src, int batch, int rows, int cols, int transpose, void *codes,
                    void *scales, moe_stream_t stream);

/* S0 in the layer's own terms: the MXFP8 codes of the layer's stacked expert
 * weights, one bf16 master matrix [rows, cols] per expert (cfg->E of them,
 * back to back at w_bf16).
 *   blocks_along_rows = 0: the forward operand, blocks of 32 along cols
 *     (W_gu [E*2m, d] with rows = 2m, cols = d; W_dn [E*d, m]): as
 *     moe_quantize_mx(w_bf16, cfg->E, rows, cols, 0, ...).
 *   blocks_along_rows = 1: the backward operand, each expert's matrix
 *     transposed and quantised in blocks of 32 along its rows (W_gu^T
 *     [E*d, 2m], W_dn^T [E*m, d]): as moe_quantize_mx(..., 1, ...).
 * cfg must be a valid MXFP8 config (MOE_ERR_ARG otherwise); rows and cols
 * multiples of 128; inputs finite.  Asynchronous on `stream`. */
int moe_quantize_weights(const moe_config *cfg, const void *w_bf16, int rows, int cols, int blocks_along_rows,
                         void *codes, void *scales, moe_stream_t stream);

/* S0 for a training layer: both orientations from one read of the bf16
 * masters.  codes/scales exactly as moe_quantize_mx(transpose = 0) and
 * codes_t/scales_t exactly as moe_quantize_mx(transpose = 1) would write them
 * (bit-identical, canonical scales).  rows and cols multiples of 128; inputs
 * finite. */
int moe_quantize_mx_both(const void *src, int batch, int rows, int cols, void *codes, void *scales,
                         void *codes_t, void *scales_t, moe_stream_t stream);

/* S0 for the whole layer, straight into the operands moe_forward and
 * moe_backward read (one read of each bf16 master; "Mixture-of-Kittens" wiki
 * page, Key claims, MXFP8 bullet: MXFP8 expert weights with BF16 masters).
 * w_gu [E, 2m, d] and w_dn [E, d, m] bf16 masters of cfg's experts.
 *   MXFP8: gu / dn = E4M3 codes [E*2m, d] / [E*d, m] with PREPARED scales
 *     gu_scale / dn_scale (as moe_quantize_weights(blocks_along_rows = 0)
 *     followed by moe_prepare_scales, bit for bit); with gu_t and dn_t given,
 *     also the backward operands gu_t [E*d, 2m] + gu_t_scale and dn_t [E*m, d]
 *     + dn_t_scale (blocks_along_rows = 1), from the same read of the masters.
 *   BF16: the masters are the forward operands (copied into gu / dn when
 *     those name other buffers; NULL = use the masters); with gu_t and dn_t
 *     given, the per-expert transposes of the masters (the *_scale pointers are
 *     unused).
 *   NVFP4: gu / dn = packed codes [E*2m, d/2] / [E*d, m/2] with prepared
 *     scales and the experts' second-level scales gu_gscale / dn_gscale [E]
 *     fp32 (2688 / the expert matrix's amax); no backward operands.
 * gu_t and dn_t are both NULL (forward only) or both given (MOE_ERR_ARG
 * otherwise).  gu_gscale / dn_gscale are required with NVFP4 (4-byte
 * aligned suffices: they hold one fp32 per expert) and ignored otherwise.
 * Re-run after every update of the masters.  Asynchronous on `stream`. */
int moe_prepare_weights(const moe_config *cfg, const void *w_gu, const void *w_dn, void *gu, void *gu_scale,
                        void *dn, void *dn_scale, void *gu_t, void *gu_t_scale, void *dn_t, void *dn_t_scale,
                        float *gu_gscale, float *dn_gscale, moe_stream_t stream);

/* MXFP8 scales from the canonical order to the prepared operand layout that
 * moe_weights' *_scale fields take (a permutation of bytes, part of S0):
 * scales [rows, K/32] -> prepared (rows*K/32 bytes).  rows and K multiples of
 * 128 (MOE_ERR_SHAPE otherwise); the two buffers must not overlap
 * (MOE_ERR_ARG if they are the same pointer).  Asynchronous on `stream`. */
int moe_prepare_scales(const void *scales, int64_t rows, int32_t K, void *prepared, moe_stream_t stream);

/* The inverse of moe_prepare_scales: prepared -> canonical [rows, K/32]
 * (e.g. to read the scale buffers moe_buffer_info names, or to save prepared
 * weights in the format's own order).  Same rules. */
int moe_canonical_scales(const void *prepared, int64_t rows, int32_t K, void *scales, moe_stream_t stream);

/* Per-batch transpose of bf16 matrices: src [batch, rows, cols] ->
 * dst [batch, cols, rows] (rows, cols multiples of 32). */
int moe_transpose_bf16(const void *src, int batch, int rows, int cols, void *dst,
                       moe_stream_t stream);

/*
 * S1 + S2: router top-k and the device-side schedule (daily-ai-frontier
 * summary, TL;DR: routing fused into the layer; wiki page, flowchart and Key
 * claims: the device-side schedule kernel never talks to the host).
 * logits [T, E] fp32 (finite).  Outputs (device, caller-owned):
 *   idx [T, k] int32: experts ordered by (logit desc, index asc), first k;
 *   w [T, k] fp32: softmax over the k chosen logits (= softmax over E
 *                  renormalised to the chosen k);
 *   counts [E] int32; offsets [E+1] int32 (exclusive prefix sum);
 *   perm [T*k] int32: perm[t*k+j] = expert-sorted row of slot (t, j); rows of
 *                  one expert keep ascending slot order (stable).
 * Any output pointer may be NULL, in which case that output stays in `ws`.
 */
int moe_route(const moe_config *cfg, const float *logits, int32_t *idx, float *w, int32_t *counts,
              int32_t *offsets, int32_t *perm, void *ws, moe_stream_t stream);

/*
 * Router projection in front of the layer (daily-ai-frontier summary, TL;DR:
 * routing is the first fused stage; the pages do not define the projection,
 * so it is a bias-free linear map): logits [T, E] fp32 = x [T, d] bf16 *
 * W_r [E, d] bf16 ^T with fp32 accumulation, on the library's own tcgen05
 * GEMM (fp32 epilogue) through a zero-padded [roundup(T,128), roundup(E,128)]
 * buffer inside `ws`.  Bitwise reproducible.
 */
int moe_router_forward(const moe_config *cfg, const void *x, const void *W_r, float *logits, void *ws,
                       moe_stream_t stream);

/*
 * Router backward: dlogits [T, E] fp32 (moe_backward's output, including the
 * load-balancing term) is rounded to bf16 g; then dx [T, d] bf16 is updated in
 * place to bf16(dx + g W_r) (the layer's dx plus the router's, one rounding)
 * and dW_r [E, d] bf16 = bf16(g^T x).  Both on the library's own tcgen05 GEMM
 * (the first with an add-into-bf16 epilogue), over zero-padded copies of g,
 * g^T, W_r^T and x^T inside `ws`, which must be sized with MOE_FLAG_BACKWARD.
 */
int moe_router_backward(const moe_config *cfg, const float *dlogits, const void *x, const void *W_r, void *dx,
                        void *dW_r, void *ws, moe_stream_t stream);

/*
 * Forward pass: route -> schedule -> dispatch gather (MXFP8: x quantised in
 * the gather) -> gate/up grouped GEMM with SwiGLU (MXFP8: h quantised in the
 * epilogue) -> down grouped GEMM -> shared expert -> combine
 *     y[t] = bf16( sum_{j<k} w[t,j] * o[row(t,j)] + s[t] )   (fixed j order)
 * x [T, d] bf16; logits [T, E] fp32; y [T, d] bf16 output.
 * saved: NULL for inference, else moe_saved_bytes() bytes that the backward
 * reads.  ws: moe_workspace_bytes() bytes.
 * Expert-sorted rows are padded per expert to multiples of 128: the rows of
 * expert e occupy [poff[e], poff[e] + counts[e]) with
 * poff[e] = sum_{e'<e} roundup(counts[e'], 128).
 */
int moe_forward(const moe_config *cfg, const void *x, const float *logits, const moe_weights *W,
                void *y, void *saved, void *ws, moe_stream_t stream);

/*
 * Backward pass (wiki page, Key claims: reverse-combine, then the expert
 * GEMMs' dgrad/wgrad, then reverse-dispatch).  Inputs: dy [T, d] bf16, the
 * forward's x, weights (including the backward operands) and `saved`.
 * Outputs: dx [T, d] bf16; dlogits [T, E] fp32 (w_j (g_j - sum_i w_i g_i) at
 * the chosen experts, g_j = <dy_t, o_j>, 0 elsewhere); dW_gu [E, 2m, d] and
 * dW_dn [E, d, m] bf16, every element written (all zeros for an expert that
 * received no rows, so the buffers need no clearing beforehand); dWs_gu
 * [2m_s, d], dWs_dn [d, m_s] bf16 (shared expert; NULL when absent).
 */
int moe_backward(const moe_config *cfg, const void *dy, const void *x, const moe_weights *W,
                 const void *saved, void *dx, float *dlogits, void *dW_gu, void *dW_dn,
                 void *dWs_gu, void *dWs_dn, void *ws, moe_stream_t stream);

/*
 * Router top-k + schedule without a workspace, for callers that cannot call
 * cudaMalloc: code inside a host framework that owns every device byte through
 * its own arena, or a latency-critical path on which an allocation (which can
 * synchronise the device) is not acceptable.  The pages have no counterpart:
 * this is an extra entry point of this library, not a step of the method.
 * Computes exactly what moe_route computes (same kernels, same bits); all
 * seven pointers are required (no output can stay in a workspace).
 * Scratch: a fixed array in the library's device memory, sized for at most
 * MOE_ROUTE_NOALLOC_MAX_SLOTS routed slots (T*k) and
 * MOE_ROUTE_NOALLOC_MAX_EXPERTS experts (about 2 MiB, held by every GPU that
 * loads the library until the process exits); larger shapes return
 * MOE_ERR_SHAPE.  Every call shares that array and leaves its contents behind
 * (nothing in it needs to start at zero): calls that overlap on the GPU (on
 * different streams, or from several host threads) race and corrupt each
 * other's results.  Calls on one stream are ordered and safe.  The first call
 * on a device looks up the array's device address (cudaGetSymbolAddress); make
 * that first call before any stream capture.  The address is kept for the life
 * of the process: calls made after cudaDeviceReset (or anything else that
 * destroys and re-creates the device's primary context) are not supported.
 * Allocates nothing.
 */
#define MOE_ROUTE_NOALLOC_MAX_SLOTS 262144
#define MOE_ROUTE_NOALLOC_MAX_EXPERTS 1024
int moe_route_noalloc(const moe_config *cfg, const float *logits, int32_t *idx, float *w,
                      int32_t *counts, int32_t *offsets, int32_t *perm, moe_stream_t stream);

/* Synchronises `stream`, returns the device status word recorded in `ws`
 * (MOE_OK, MOE_ERR_TIMEOUT, or in a debug build MOE_ERR_BOUNDS; a timeout is
 * reported first when both happened) and clears it.  Returns MOE_ERR_CUDA if
 * the stream reports a CUDA error. */
int moe_get_status(void *ws, moe_stream_t stream);

/* Static description of a status code (never NULL). */
const char *moe_status_string(int status);

/*
 * Optional per-launch timing (process-wide, for benchmarks and profilers).
 * moe_trace_enable(n) creates n pairs of CUDA events (n = 0 disables tracing
 * and destroys them); while enabled, every kernel launch made by moe_route,
 * moe_forward and moe_backward is bracketed by an event pair recorded on the
 * call's stream, in launch order, until n launches are recorded.  Tracing
 * adds two event records per launch and changes nothing else.
 * moe_trace_clear() restarts at slot 0; moe_trace_count() is the number of
 * recorded launches; moe_trace_name(i) names launch i (static string, NULL
 * when i is out of range); moe_trace_ms(i) synchronises on launch i's end
 * event and returns its duration in milliseconds (negative on error).
 * Not thread-safe: trace from one host thread.
 */
int moe_trace_enable(int capacity);
void moe_trace_clear(void);
int moe_trace_count(void);
const char *moe_trace_name(int i);
float moe_trace_ms(int i);

#ifdef __cplusplus
}
#endif

#endif /* MOE_H */
