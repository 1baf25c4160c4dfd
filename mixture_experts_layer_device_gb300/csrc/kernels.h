// Internal launchers of the layer's kernels (host side).  All launches are
// asynchronous on the given stream; each returns cudaGetLastError().
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace moe {

// Device status word bits (kept in the workspace, read by moe_get_status).
constexpr int kStatusTimeout = 1;
constexpr int kStatusBounds = 2;  // a debug-build bounds check failed
// Default limit of every device-side wait.
constexpr unsigned long long kWaitTimeoutNs = 4000000000ull;

// Chunk of flat slots handled by one warp in the schedule kernels.
constexpr int kSchedChunk = 1024;

struct RouteBufs {
  int *idx;       // [T*k]
  float *w;       // [T*k]
  int *counts;    // [E]
  int *offsets;   // [E+1]
  int *perm;      // [R]  slot -> row
  int *inv;       // [R]  row -> slot
  int *poff;      // [E+1] padded offsets (multiples of 128)
  int *hist;      // [nchunks * E] scratch
  int *tile_order;  // [Rp / 32] processing order of 32-row tiles (may be NULL: row order)
  // extents and the status word for the bounds checks of debug builds
  int n_tok;      // T
  long n_slots;   // T * k
  long n_rows;    // padded rows Rp
  int *status;    // may be NULL (nothing recorded)
};

cudaError_t launch_route(const float *logits, int T, int E, int k, const RouteBufs &b,
                         cudaStream_t s);

// Gather routed rows of x into padded expert-sorted order (zero padding rows).
// MX: when xs is not NULL, writes the row-blocked codes of each routed row to
// xs [Rp, d] with tiled scales (K = d); when xT is not NULL, also the
// column-blocked transposed codes xT [d, Rp] (+ tiled scales, K = Rp) of the
// same rows.  Without xT (inference) every token is first quantised once into
// xq [T, d] (canonical scales xq_sf [T, d / 32]) and the dispatch copies those
// codes; with xT the row codes are encoded from the bf16 rows it reads anyway.
// BF16: copies rows of x to xs.
cudaError_t launch_gather(const void *x, int T, int d, int k, int E, const RouteBufs &b,
                          int64_t rp_max, bool mx, void *xs, uint8_t *xs_sf, uint8_t *xT, uint8_t *xT_sf,
                          uint8_t *xq, uint8_t *xq_sf, cudaStream_t s);

// y[t] = bf16( sum_j w[t,j] * o[row(t,j)] + s[t] ), fixed j order.
cudaError_t launch_combine(const void *o, const void *s_out, int T, int d, int k, int E,
                           const RouteBufs &b, void *y, cudaStream_t s);

// Reverse combine, BF16 experts: dO[row] = bf16(w * dy[t]) (zero on padding
// rows), g[slot] = <dy[t], o[row]>.
cudaError_t launch_reverse_combine(const void *dy, const void *o, int T, int d, int k, int E,
                                   const RouteBufs &b, int64_t rp_max, void *dO, float *g, cudaStream_t s);

// Reverse combine, MXFP8, fused with the wgrad operand: g[slot] = <dy[t], o[row]>,
// dO = bf16(w * dy) written as row-blocked codes dOq [Rp, d] (+ tiled scales,
// K = d) and column-blocked transposed codes dOT [d, ld_t = Rp] (+ tiled
// scales, K = Rp); padding rows give zero codes.
cudaError_t launch_reverse_combine_mx(const void *dy, const void *o, int T, int d, int k, int E,
                                      const RouteBufs &b, int64_t rp_max, float *g, uint8_t *dOq,
                                      uint8_t *dOq_sf, uint8_t *dOT, uint8_t *dOT_sf, cudaStream_t s);

// Reverse dispatch: dx[t] = bf16( sum_j dX[row(t,j)] + dxs[t] ); dlogits row
// (+ aux_grad row when given: the load-balancing term's gradient).
cudaError_t launch_reverse_dispatch(const void *dX, const void *dxs, const float *g, int T,
                                    int d, int k, int E, const RouteBufs &b, void *dx,
                                    float *dlogits, const float *aux_grad, cudaStream_t s);

// Transpose of a row block: src [*, C] (row stride C) -> dst [C, ld_dst],
// dst[c][r] = src[row(r)][c] for r < nrows (device count *nrows_dev when not
// NULL, else nrows_out, a multiple of 32).  With `gather`, row(r) is the token
// of padded expert row r (x re-gathered; -1 on padding rows), else row(r) = r;
// rows with row(r) < 0 or row(r) >= nsrc read as zero.  bf16 output (the BF16
// wgrad operands; MXFP8 ones are written by the kernels that produce them).
cudaError_t launch_transpose_rows(const void *src, int C, int nrows_out, const int *nrows_dev,
                                  long nsrc, bool gather, int k, int E, const RouteBufs *b,
                                  int64_t rows_alloc, void *dst, int64_t ld_dst, cudaStream_t s);

// Weight preparation: scales canonical [rows, K/32] (canon) or in the tiled
// operand layout the GEMMs read.
cudaError_t launch_quantize_mx(const void *src, int batch, int rows, int cols, bool transpose,
                               uint8_t *codes, uint8_t *scales, bool canon, cudaStream_t s);
cudaError_t launch_transpose_bf16(const void *src, int batch, int rows, int cols, void *dst,
                                  cudaStream_t s);

// ---------------------------------------------------------------- GEMM
enum GemmSched { SCHED_GROUP_M = 0, SCHED_DENSE = 1, SCHED_GROUP_K = 2 };
// Operand formats of launch_gemm.
enum GemmFmt { FMT_BF16 = 0, FMT_MXFP8 = 1, FMT_NVFP4 = 2 };

// EPI_STORE_F32: fp32 output (the router logits); EPI_ADD_BF16: out = bf16(out +
// acc) with `out` read back through aux (the router's dx contribution).  Both
// run on the single-CTA kernel only.
enum GemmEpi { EPI_STORE = 0, EPI_SWIGLU = 1, EPI_SWIGLU_BWD = 2, EPI_STORE_F32 = 3, EPI_ADD_BF16 = 4 };

// MXFP8 scales [rows, K/32] canonical -> tiled operand layout (to_tiled) or back;
// rows and K multiples of 128.
cudaError_t launch_scales_layout(const void *src, long rows, int K, bool to_tiled, void *dst, cudaStream_t s);

// Both MXFP8 orientations of bf16 weights [batch, rows, cols] from one read:
// codes/scales as launch_quantize_mx(transpose = false), codes_t/scales_t as
// launch_quantize_mx(transpose = true).
cudaError_t launch_quantize_mx_both(const void *src, int batch, int rows, int cols, uint8_t *codes,
                                    uint8_t *scales, uint8_t *codes_t, uint8_t *scales_t, bool canon,
                                    cudaStream_t s);

// Load-balancing term (Switch-style, over the routed slots): per-block partial
// sums of the full softmax (part [balance_blocks(T), E]), the gradient rows
// [T, E] (grad, may be NULL) and out = [loss, P[E], f[E]], all fp32 and
// bitwise reproducible.
constexpr int kBalanceTokensPerBlock = 64;
int balance_blocks(int T);
cudaError_t launch_balance(const float *logits, int T, int E, int k, const int *counts, float alpha, float *part,
                           float *grad, float *out, cudaStream_t s);
// dst[i] = bf16(src[i]) (round to nearest even), n values.
cudaError_t launch_to_bf16(const float *src, long n, void *dst, cudaStream_t s);
// dst [rows_p, cols_p] bf16 = bf16(src [rows, cols] fp32), zero beyond rows / cols
// (cols_p a multiple of 8).
cudaError_t launch_pad_to_bf16(const float *src, int rows, int cols, int rows_p, int cols_p, void *dst,
                               cudaStream_t s);
// dst [rows, cols] fp32 = the top-left corner of src [*, ld_src] fp32.
cudaError_t launch_crop_f32(const float *src, int rows, int cols, long ld_src, float *dst, cudaStream_t s);

// NVFP4 second-level scales of `batch` bf16 tensors of n values each (n a
// multiple of 8): gscale[t] = 2688 / amax(|tensor t|), 1 for an all-zero one.
cudaError_t launch_nv_global_scales(const void *src, int batch, long n, float *gscale, cudaStream_t s);
// NVFP4 rows src [rows, cols] bf16 (cols a multiple of 64) -> packed codes
// [rows, cols / 2] and scale codes (tiled operand layout with K' = 2 cols, or
// canonical [rows, cols / 16]); row r's tensor has second-level scale
// gscale[r / rows_per_tensor].
cudaError_t launch_nv_quantize_rows(const void *src, long rows, int cols, long rows_per_tensor, const float *gscale,
                                    uint8_t *codes, uint8_t *scales, bool tiled, cudaStream_t s);
// NVFP4 dispatch: padded expert-sorted rows [0, rows) <- their tokens' codes
// (xq [T, d / 2], canonical scales [T, d / 16]), tiled scales (K' = 2 d).
cudaError_t launch_nv_gather(const uint8_t *xq, const uint8_t *xq_sf, int d, int k, int E, const RouteBufs &b,
                             long rows, uint8_t *xs, uint8_t *xs_sf, cudaStream_t s);

// Row-blocked MXFP8 codes of every token: x [T, d] bf16 -> codes [T, d] and
// canonical scales [T, d/32] (the ring dispatch gathers these rows).
cudaError_t launch_quantize_tokens(const void *x, int T, int d, uint8_t *codes, uint8_t *scales,
                                   cudaStream_t s);

// Persistent ring dispatch (S3 fused with the MXFP8 gate/up GEMM): the first
// `gather_ctas` CTAs of the launch gather and quantise 128-row tiles of
// expert-sorted rows into a ring of `slots` tiles; the other CTAs run the GEMM
// on the ring.  Tile u (padded rows [128u, 128u + 128)) goes to slot u % slots.
struct RingArgs {
  const uint8_t *xq;     // [T, d] row-blocked codes of every token (launch_quantize_tokens)
  const uint8_t *xq_sf;  // [T, d/32] their scales, canonical order
  RouteBufs rb;          // route / schedule arrays (token of each row)
  int k;
  int slots;          // ring capacity in 128-row tiles
  int gather_ctas;    // CTAs of the launch that gather (the rest compute)
  uint8_t *codes;     // [slots * 128, d] E4M3 codes: the GEMM's A operand
  uint8_t *sf;        // tiled scales of `codes` (K = d)
  int *ready;         // [slots] index + 1 of the tile last published in the slot
  int *freed;         // [slots] GEMM tiles whose loads from the slot have landed (cumulative)
  int *abort;         // launch-wide abort word (set when any wait runs out)
};

struct GemmArgs {
  int sched;
  int E;              // groups (experts); 1 for dense
  const int *poff;    // [E+1] padded offsets (GROUP_M: A rows; GROUP_K: K ranges)
  int M;              // DENSE: rows of A; GROUP_K: rows of A (= output rows per group)
  int K;              // GROUP_M / DENSE: reduction length; GROUP_K with poff == NULL: K
  int n_tiles;        // output column tiles
  int b_rows_per_group;  // GROUP_M: rows of B per expert
  int b_split;        // SWIGLU: row offset of the up half inside an expert's B (m); else 0
  // MX scales (tiled layout), K groups of 128 per 128-row group
  const uint8_t *sfa;
  int sfa_kg;
  const uint8_t *sfb;
  int sfb_kg;
  // epilogue
  void *out;          // bf16 output (STORE: D; SWIGLU: h; SWIGLU_BWD: dGU)
  long ldo;
  void *out2;         // SWIGLU: G|U save [rows, 2m] bf16 (may be NULL)
  long ldo2;
  long out_rows;      // rows of out / out2 / outq (stores beyond are skipped)
  uint8_t *outq;      // SWIGLU / SWIGLU_BWD MX codes (may be NULL)
  uint8_t *outq_sf;   // tiled scales of outq
  long ldq;           // row stride of outq (= its K)
  uint8_t *outT;      // MXFP8 training, column-blocked codes (may be NULL): SWIGLU h^T [m, ldT],
                      // SWIGLU_BWD dGU^T [2m, ldT]
  uint8_t *outT_sf;   // tiled scales of outT (K = ldT)
  long ldT;           // row stride of outT (padded rows)
  const void *aux;    // SWIGLU_BWD: saved G|U bf16
  long ld_aux;
  int m_half;         // SWIGLU / SWIGLU_BWD: m
  long sfa_bytes, sfb_bytes;  // sizes of the scale buffers (bounds checks of debug builds)
  const float *a_gscale;  // NVFP4: second-level scale of A (one value; NULL = 1)
  const float *b_gscale;  // NVFP4: second-level scale of B per group [E]
  float *dump;        // SWIGLU (tests): fp32 h before quantisation [rows, ld_dump] (may be NULL)
  long ld_dump;
  int skip_empty;     // GROUP_K: tiles with an empty reduction are left to launch_zero_empty_experts
  int *status;
  unsigned long long timeout_ns;  // limit of every wait in the launch
  int debug_starve;   // test hook: the producer issues no loads (the MMA wait runs out);
                      // with a ring, the gather CTAs publish nothing instead
  RingArgs ring;      // launch_gemm_ring only
};

// Zeros for the weight gradients of experts that received no rows: dW holds E
// matrices of expert_bytes (a multiple of 16) each; expert e's is cleared when
// counts[e] == 0.  Plain 16-byte stores from a grid of 1 MB pieces.
cudaError_t launch_zero_empty_experts(void *dW, int E, long expert_bytes, const int *counts, cudaStream_t s);

// D = A * B^T with A [rows, K] and B [rows, K] K-major (TMA maps built by the
// caller, box = 128 rows x 128 bytes, 128-byte swizzle); bn = 128 or 256
// output columns per tile; `grid` persistent CTAs (<= number of SMs).  The
// epilogue writes args.out / out2 / outq (row strides ldo / ldo2 / ldq) with
// coalesced global stores, rows < args.out_rows.
cudaError_t launch_gemm(int fmt, int bn, int epi, const CUtensorMap &ta, const CUtensorMap &tb,
                        const GemmArgs &args, int grid, cudaStream_t s);

// The MXFP8 gate/up GEMM with SwiGLU epilogue fed by the ring (args.ring):
// one cooperative launch of `grid` CTAs (all co-resident, one per SM), of
// which args.ring.gather_ctas gather.  `ta` maps the ring codes
// [slots * 128, d].  args.ring.ready / freed / abort must be zero at launch.
cudaError_t launch_gemm_ring(const CUtensorMap &ta, const CUtensorMap &tb, const GemmArgs &args, int grid,
                             cudaStream_t s);
// CTAs of the ring GEMM that can be resident at once on the current device.
int ring_max_ctas();

// Tensor maps of one 2-CTA GEMM launch: operands (box 128 rows x 128 bytes,
// 128-byte swizzle) and MXFP8 scale buffers viewed as rows of 256 bytes (box
// 2 rows = one 512-byte atom).
struct PairMaps {
  CUtensorMap a, b, sfa, sfb;
};

// D = A * B^T on CTA pairs (tcgen05 cta_group::2): 256 x 256 tiles, two
// consecutive 128-row M-tiles of one group per pair.  Requires N tiles of 256
// and, for SCHED_GROUP_K, M a multiple of 256.  `clusters` pairs are launched
// (<= pair_max_clusters()).
cudaError_t launch_gemm_pair(bool mx, int epi, const PairMaps &maps, const GemmArgs &args,
                             int clusters, cudaStream_t s);
int pair_max_clusters(bool mx, int epi);

}  // namespace moe
