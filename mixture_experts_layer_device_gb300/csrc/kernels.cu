// Memory-bound kernels of the layer: router top-k, the device-side schedule
// (histogram, scan, stable permutation), dispatch gather with fused MXFP8
// quantisation, deterministic combine, reverse combine / reverse dispatch of
// the backward pass, transposes and weight quantisation.
//
// Method references ("Mixture-of-Kittens" pages):
//   routing fused into the layer            -- daily-ai-frontier summary, TL;DR
//   device-side schedule, no CPU sync        -- wiki page, flowchart + Key claims
//   quantisation fused into dispatch          -- wiki page, Key claims (MXFP8)
//   fixed-order (bitwise deterministic) sum  -- wiki page, TL;DR + Key claims
//   reverse-combine / reverse-dispatch       -- wiki page, Key claims (directions)
#include <cuda_bf16.h>
#include <math.h>

#include "common.cuh"
#include "dispatch_tile.cuh"
#include "kernels.h"

namespace moe {

namespace {

// ------------------------------------------------------------ S1: route
// One warp per token.  Top-k by repeated warp argmax under the total order
// (logit descending, index ascending); weights = softmax over the k chosen
// logits, summed in slot order.

// An unsigned key that orders like the fp32 value (a > b exactly when key(a) >
// key(b)); -0 is first made +0, so equal values get equal keys.
MOE_DEV uint32_t order_key(float v) {
  const uint32_t u = __float_as_uint(v + 0.0f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
MOE_DEV float key_value(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

template <int VPL>
__global__ void __launch_bounds__(256) route_topk_kernel(const float *__restrict__ logits, int T,
                                                         int E, int k, int *__restrict__ idx,
                                                         float *__restrict__ w) {
  const int t = static_cast<int>((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (t >= T) return;
  const float *row = logits + static_cast<size_t>(t) * E;
  float v[VPL];
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    const int e = lane + 32 * i;
    v[i] = e < E ? __ldg(row + e) : -INFINITY;
  }
  uint32_t taken = 0;
  int my_e = 0;
  float my_l = 0.f;
  for (int j = 0; j < k; ++j) {
    float bv = -INFINITY;
    int be = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
      const int e = lane + 32 * i;
      const bool ok = e < E && !((taken >> i) & 1u);
      if (ok && (v[i] > bv || (v[i] == bv && e < be))) {
        bv = v[i];
        be = e;
      }
    }
    // warp argmax: the largest key, then the smallest expert among the lanes holding it
    const uint32_t kv = order_key(bv);
    const uint32_t km = __reduce_max_sync(0xffffffffu, kv);
    be = static_cast<int>(__reduce_min_sync(0xffffffffu, kv == km ? static_cast<uint32_t>(be) : 0xffffffffu));
    bv = key_value(km);
    if ((be & 31) == lane) taken |= 1u << (be >> 5);
    if (lane == j) {
      my_e = be;
      my_l = bv;
    }
  }
  const float l0 = __shfl_sync(0xffffffffu, my_l, 0);
  const float ex = lane < k ? expf(my_l - l0) : 0.f;
  float sum = 0.f;
  for (int j = 0; j < k; ++j) sum += __shfl_sync(0xffffffffu, ex, j);
  if (lane < k) {
    idx[static_cast<size_t>(t) * k + lane] = my_e;
    w[static_cast<size_t>(t) * k + lane] = ex / sum;
  }
}

// ------------------------------------------------------------ S2: schedule
// (a) per-chunk expert histograms (integer counts: order-independent).
__global__ void __launch_bounds__(128) sched_hist_kernel(const int *__restrict__ idx, int R, int E,
                                                         int nchunks, int *__restrict__ hist, int *status) {
  extern __shared__ int cnt[];
  const int wib = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = blockIdx.x * (blockDim.x >> 5) + wib;
  int *my = cnt + wib * E;
  if (c >= nchunks) return;
  for (int e = lane; e < E; e += 32) my[e] = 0;
  __syncwarp();
  const int base = c * kSchedChunk;
  for (int i = lane; i < kSchedChunk; i += 32) {
    const int s = base + i;
    if (s < R) {
      const int e = __ldg(idx + s);
      if (MOE_BOUNDS_OK(e >= 0 && e < E, status)) atomicAdd(&my[e], 1);
    }
  }
  __syncwarp();
  for (int e = lane; e < E; e += 32) hist[static_cast<size_t>(c) * E + e] = my[e];
}

MOE_DEV int block_exclusive_scan(int v, int *warp_tot, int *total) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  int inc = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(0xffffffffu, inc, off);
    if (lane >= off) inc += o;
  }
  if (lane == 31) warp_tot[wid] = inc;
  __syncthreads();
  if (wid == 0) {
    const int nw = blockDim.x >> 5;
    int x = lane < nw ? warp_tot[lane] : 0;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, x, off);
      if (lane >= off) x += o;
    }
    if (lane < nw) warp_tot[lane] = x - (lane < nw ? warp_tot[lane] : 0);  // exclusive
    if (lane == nw - 1) *total = x;
  }
  __syncthreads();
  return inc - v + warp_tot[wid];
}

// (b) one block: per-expert exclusive prefix over chunks (in place), counts,
// offsets (exclusive scan) and 128-padded offsets.
__global__ void __launch_bounds__(1024) sched_scan_kernel(int *__restrict__ hist, int nchunks, int E,
                                                          int *__restrict__ counts,
                                                          int *__restrict__ offsets,
                                                          int *__restrict__ poff) {
  __shared__ int wt[32];
  __shared__ int tot;
  const int e = threadIdx.x;
  int total = 0;
  if (e < E) {
    // 8 chunks' counts are loaded before any is replaced by its running
    // prefix, so the loads overlap instead of forming one chain per expert.
    constexpr int U = 8;
    int c = 0;
    for (; c + U <= nchunks; c += U) {
      int v[U];
#pragma unroll
      for (int j = 0; j < U; ++j) v[j] = hist[static_cast<size_t>(c + j) * E + e];
#pragma unroll
      for (int j = 0; j < U; ++j) {
        hist[static_cast<size_t>(c + j) * E + e] = total;
        total += v[j];
      }
    }
    for (; c < nchunks; ++c) {
      const size_t p = static_cast<size_t>(c) * E + e;
      const int v = hist[p];
      hist[p] = total;
      total += v;
    }
    counts[e] = total;
  }
  const int a = e < E ? total : 0;
  const int pc = e < E ? ((total + 127) & ~127) : 0;
  const int ea = block_exclusive_scan(a, wt, &tot);
  const int ta = tot;
  __syncthreads();
  const int ep = block_exclusive_scan(pc, wt, &tot);
  if (e < E) {
    offsets[e] = ea;
    poff[e] = ep;
  }
  if (e == 0) {
    offsets[E] = ta;
    poff[E] = tot;
  }
}

// (c) one warp per chunk: stable ranks.  Slots are visited in flat order 32 at
// a time; lanes with equal experts are ranked by lane (match_any), so rows of
// an expert keep ascending slot order.
__global__ void __launch_bounds__(128) sched_scatter_kernel(const int *__restrict__ idx, int R, int E,
                                                            int nchunks,
                                                            const int *__restrict__ hist_excl,
                                                            const int *__restrict__ offsets,
                                                            int *__restrict__ perm,
                                                            int *__restrict__ inv, int *status) {
  extern __shared__ int cnt[];
  const int wib = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = blockIdx.x * (blockDim.x >> 5) + wib;
  if (c >= nchunks) return;
  int *my = cnt + wib * E;
  for (int e = lane; e < E; e += 32) my[e] = offsets[e] + hist_excl[static_cast<size_t>(c) * E + e];
  __syncwarp();
  const int base = c * kSchedChunk;
  for (int it = 0; it < kSchedChunk; it += 32) {
    const int s = base + it + lane;
    int e = s < R ? __ldg(idx + s) : -1;
    if (s < R && !MOE_BOUNDS_OK(e >= 0 && e < E, status)) e = -1;
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const int rank = __popc(peers & ((1u << lane) - 1u));
    const int row = e >= 0 ? my[e] + rank : 0;
    __syncwarp();
    if (e >= 0 && rank == 0) my[e] += __popc(peers);
    __syncwarp();
    if (e >= 0 && MOE_BOUNDS_OK(row >= 0 && row < R, status)) {
      perm[s] = row;
      inv[row] = s;
    }
  }
}

// ------------------------------------------------------------ S3: dispatch
// BF16: one warp per padded row copies its token's row of x (zeros for padding rows).
__global__ void __launch_bounds__(256) gather_bf16_kernel(const uint4 *__restrict__ x, int d, int k, int E,
                                                          RouteBufs b, int64_t rp_max, uint4 *__restrict__ xs) {
  const int64_t pr = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (pr >= rp_max || pr >= __ldg(b.poff + E)) return;
  const int tok = token_of_row(b, E, k, static_cast<int>(pr), nullptr);
  const int vec = d >> 3;
  const uint4 *src = x + static_cast<size_t>(tok < 0 ? 0 : tok) * vec;
  for (int i = lane; i < vec; i += 32)
    xs[static_cast<size_t>(pr) * vec + i] = tok >= 0 ? __ldg(src + i) : make_uint4(0, 0, 0, 0);
}

// MXFP8 dispatch as 32-row tiles: rows of x (by token) are quantised along d
// into xs codes [Rp, d] (+ tiled scales, K = d) and, when xT is given, the
// block's 32 rows are also quantised per column into the transposed codes
// xT [d, ld_t] (+ tiled scales, K = ld_t): the wgrad operand of the backward.
// Processing order of the 32-row tiles of the expert-sorted rows, for the
// kernels that read one token row per routed row (MXFP8 dispatch and reverse
// combine): tiles sorted by the token of their first row, by a counting sort
// over kOrderBuckets token ranges (all-padding tiles last).  Tiles of
// different experts that hold the same tokens then run at about the same
// time, and the token rows they share come from L2 instead of HBM; in expert
// order every hot expert sweeps all T token rows again.  Only the order in
// which blocks take tiles changes: each tile is still written by one block,
// with the same values.  One block of kOrderBuckets threads.
constexpr int kOrderBuckets = 1024;

__global__ void __launch_bounds__(kOrderBuckets) tile_order_kernel(RouteBufs b, int T, int E, int k,
                                                                   int *__restrict__ order) {
  __shared__ int cnt[kOrderBuckets];
  __shared__ int wsum[kOrderBuckets / 32];
  const int tid = static_cast<int>(threadIdx.x);
  const int lane = tid & 31, warp = tid >> 5;
  const int ntiles = __ldg(b.poff + E) >> 5;
  auto key = [&](int t) {
    const int tok = token_of_row(b, E, k, t * 32, nullptr);
    return tok < 0 ? kOrderBuckets - 1
                   : static_cast<int>(static_cast<long long>(tok) * kOrderBuckets / T);
  };
  cnt[tid] = 0;
  __syncthreads();
  for (int t = tid; t < ntiles; t += kOrderBuckets) atomicAdd(&cnt[key(t)], 1);
  __syncthreads();
  // exclusive scan of the bucket counts, one bucket per thread
  const int v = cnt[tid];
  int x = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, off);
    if (lane >= off) x += y;
  }
  if (lane == 31) wsum[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = wsum[lane];
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, off);
      if (lane >= off) w += y;
    }
    wsum[lane] = w;
  }
  __syncthreads();
  cnt[tid] = x - v + (warp > 0 ? wsum[warp - 1] : 0);  // first position of the bucket
  __syncthreads();
  for (int t = tid; t < ntiles; t += kOrderBuckets) order[atomicAdd(&cnt[key(t)], 1)] = t;
}

// First row of the tile block `blk` takes, or -1 past the last tile.
MOE_DEV int tile_row0(const RouteBufs &b, int E, int blk) {
  if (blk >= (__ldg(b.poff + E) >> 5)) return -1;
  return 32 * (b.tile_order ? __ldg(b.tile_order + blk) : blk);
}

template <bool COPY>
__global__ void __launch_bounds__(256, 4) gather_mx_tile_kernel(const uint16_t *__restrict__ x,
                                                                const uint8_t *__restrict__ xq,
                                                                const uint8_t *__restrict__ xq_sf, int d, int k,
                                                                int E, RouteBufs b, uint8_t *__restrict__ xs,
                                                                uint8_t *__restrict__ xs_sf,
                                                                uint8_t *__restrict__ xT,
                                                                uint8_t *__restrict__ xT_sf, long ld_t) {
  __shared__ __align__(16) uint16_t tile[2][32][256];
  const int r0 = tile_row0(b, E, static_cast<int>(blockIdx.x));
  if (r0 < 0) return;
  dispatch_rows32<COPY>(x, xq, xq_sf, d, k, E, b, r0, xs, xs_sf, xT, xT_sf, ld_t, tile,
                        static_cast<int>(threadIdx.x));
}

// ------------------------------------------------------------ S6: combine
__global__ void __launch_bounds__(256) combine_kernel(const uint4 *__restrict__ o,
                                                      const uint4 *__restrict__ s_out, int T, int d,
                                                      int k, int E, RouteBufs b,
                                                      uint4 *__restrict__ y) {
  const int t = static_cast<int>((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (t >= T) return;
  int my_row = 0;
  float my_w = 0.f;
  if (lane < k) {
    const int slot = t * k + lane;
    const int e = __ldg(b.idx + slot);
    if (MOE_BOUNDS_OK(e >= 0 && e < E, b.status)) {
      my_row = __ldg(b.poff + e) + __ldg(b.perm + slot) - __ldg(b.offsets + e);
      my_w = __ldg(b.w + slot);
      if (!MOE_BOUNDS_OK(my_row >= 0 && my_row < b.n_rows, b.status)) my_row = 0, my_w = 0.f;
    }
  }
  const int vec = d >> 3;
  for (int i = lane; i < vec; i += 32) {
    float acc[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) acc[q] = 0.f;
    for (int j = 0; j < k; ++j) {
      const int row = __shfl_sync(0xffffffffu, my_row, j);
      const float wj = __shfl_sync(0xffffffffu, my_w, j);
      float f[8];
      unpack8(__ldg(o + static_cast<size_t>(row) * vec + i), f);
#pragma unroll
      for (int q = 0; q < 8; ++q) acc[q] = fmaf(wj, f[q], acc[q]);
    }
    if (s_out) {
      float f[8];
      unpack8(__ldg(s_out + static_cast<size_t>(t) * vec + i), f);
#pragma unroll
      for (int q = 0; q < 8; ++q) acc[q] += f[q];
    }
    y[static_cast<size_t>(t) * vec + i] = pack8(acc);
  }
}

// ------------------------------------------------------------ B1: reverse combine (BF16 experts)
__global__ void __launch_bounds__(256) reverse_combine_kernel(
    const uint4 *__restrict__ dy, const uint4 *__restrict__ o, int d, int k, int E, RouteBufs b,
    int64_t rp_max, uint4 *__restrict__ dO, float *__restrict__ g) {
  const int64_t pr = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (pr >= rp_max || pr >= __ldg(b.poff + E)) return;
  int slot = 0;
  const int tok = token_of_row(b, E, k, static_cast<int>(pr), &slot);
  const float wv = tok >= 0 ? __ldg(b.w + slot) : 0.f;
  const int vec = d >> 3;
  float dot = 0.f;
  for (int i = lane; i < vec; i += 32) {
    float f[8];
    if (tok >= 0) {
      float fy[8], fo[8];
      unpack8(__ldg(dy + static_cast<size_t>(tok) * vec + i), fy);
      unpack8(__ldg(o + static_cast<size_t>(pr) * vec + i), fo);
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        dot = fmaf(fy[q], fo[q], dot);
        f[q] = round_bf16(wv * fy[q]);
      }
    } else {
#pragma unroll
      for (int q = 0; q < 8; ++q) f[q] = 0.f;
    }
    dO[static_cast<size_t>(pr) * vec + i] = pack8(f);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
  if (tok >= 0 && lane == 0) g[slot] = dot;
}

// ------------------------------------------------------------ B1, MXFP8: fused
// Block: 32 padded rows x all d columns, swept in 256-column chunks with the
// next chunk's loads in flight.  Per element dO = bf16(w * dy); written as
// row-blocked E4M3 codes (the dgrad operand, blocks of 32 along d, encoded by
// the 4 threads holding a block) and, through a shared-memory tile of the
// chunk (two buffers, one barrier per chunk), as column-blocked codes of dO^T
// (the wgrad operand, one 32-row block per column, encoded by the thread
// owning the column).  g = <dy, o> per row is accumulated per thread in column
// order and reduced over the row's 8 threads in a fixed shuffle order.
__global__ void __launch_bounds__(256, 3) reverse_combine_mx_kernel(
    const uint16_t *__restrict__ dy, const uint16_t *__restrict__ o, int d, int k, int E, RouteBufs b,
    float *__restrict__ g, uint8_t *__restrict__ dOq, uint8_t *__restrict__ dOq_sf,
    uint8_t *__restrict__ dOT, uint8_t *__restrict__ dOT_sf, long ld_t) {
  __shared__ __align__(16) uint16_t tile[2][32][256];
  const int r0 = tile_row0(b, E, static_cast<int>(blockIdx.x));
  if (r0 < 0) return;
  const int tid = static_cast<int>(threadIdx.x);
  const int rr = tid >> 3;
  const int cc = (tid & 7) * 8;
  const int pr = r0 + rr;
  int slot = 0;
  const int tok = token_of_row(b, E, k, pr, &slot);
  const float wv = tok >= 0 ? __ldg(b.w + slot) : 0.f;
  const uint16_t *dyr = dy + static_cast<size_t>(tok < 0 ? 0 : tok) * d;
  const uint16_t *orow = o + static_cast<size_t>(pr) * d;
  auto load = [&](int cb, uint4 *qy, uint4 *qo) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const bool ok = tok >= 0 && cb < d;
      const size_t col = static_cast<size_t>(cb + 64 * j + cc);
      qy[j] = ok ? __ldg(reinterpret_cast<const uint4 *>(dyr + col)) : make_uint4(0, 0, 0, 0);
      qo[j] = ok ? __ldg(reinterpret_cast<const uint4 *>(orow + col)) : make_uint4(0, 0, 0, 0);
    }
  };
  uint4 qy[4], qo[4], ny[4], no[4];
  load(0, qy, qo);
  float dot = 0.f;
  int buf = 0;
  for (int cb = 0; cb < d; cb += 256) {
    load(cb + 256, ny, no);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      float fy[8], fo[8], f[8];
      unpack8(qy[j], fy);
      unpack8(qo[j], fo);
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        dot = fmaf(fy[q], fo[q], dot);
        f[q] = wv * fy[q];
      }
      const uint4 pk = pack8(f);  // dO = bf16(w * dy), one conversion per pair
      unpack8(pk, f);
      const int col = cb + 64 * j + cc;
      uint32_t byte;
      const uint2 code = mx_encode8_quad(f, &byte);
      *reinterpret_cast<uint2 *>(dOq + static_cast<size_t>(pr) * d + col) = code;
      if ((tid & 3) == 0) dOq_sf[sf_tiled_offset(pr, col >> 5, d)] = static_cast<uint8_t>(byte);
      *reinterpret_cast<uint4 *>(&tile[buf][rr][tcol(rr, 64 * j + cc)]) = pk;
    }
    __syncthreads();
    column_block_codes(tile[buf], tid, cb, r0, dOT, dOT_sf, ld_t);
    buf ^= 1;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      qy[j] = ny[j];
      qo[j] = no[j];
    }
  }
  // g: the 8 threads of a row are lanes 8u..8u+7 of one warp
#pragma unroll
  for (int off = 4; off > 0; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
  if ((tid & 7) == 0 && tok >= 0) g[slot] = dot;
}

// ------------------------------------------------------------ load-balancing term
// Warp per token: the softmax over all E experts, p = exp(l - max) / sum, with
// the max and the sum reduced by a fixed xor tree.  Each warp adds its tokens'
// p in token order; the block's 8 warp sums are added in warp order into the
// block's partial P, so P is bitwise reproducible.  With the schedule's counts
// the token's gradient row alpha E / T * p (f - sum_e f_e p_e) is written too.
template <int VPL>
__global__ void __launch_bounds__(256) balance_kernel(const float *__restrict__ logits, int T, int E, int k,
                                                      const int *__restrict__ counts, float alpha, int tpb,
                                                      float *__restrict__ part, float *__restrict__ grad) {
  extern __shared__ float wsum[];  // [8][E]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const float inv_slots = 1.0f / (static_cast<float>(T) * static_cast<float>(k));
  const float c = alpha * static_cast<float>(E) / static_cast<float>(T);
  float acc[VPL], f[VPL];
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    const int e = lane + 32 * i;
    acc[i] = 0.f;
    f[i] = e < E ? static_cast<float>(__ldg(counts + e)) * inv_slots : 0.f;
  }
  const int t0 = blockIdx.x * tpb;
  for (int tt = warp; tt < tpb; tt += 8) {
    const int t = t0 + tt;
    if (t >= T) break;
    const float *row = logits + static_cast<size_t>(t) * E;
    float v[VPL];
    float mx = -INFINITY;
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
      const int e = lane + 32 * i;
      v[i] = e < E ? __ldg(row + e) : -INFINITY;
      mx = fmaxf(mx, v[i]);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    float sum = 0.f;
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
      v[i] = (lane + 32 * i) < E ? expf(v[i] - mx) : 0.f;
      sum += v[i];
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
    float fs = 0.f;
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
      v[i] = v[i] / sum;  // p
      acc[i] += v[i];
      fs = fmaf(f[i], v[i], fs);
    }
    if (grad) {
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) fs += __shfl_xor_sync(0xffffffffu, fs, off);
      float *grow = grad + static_cast<size_t>(t) * E;
#pragma unroll
      for (int i = 0; i < VPL; ++i) {
        const int e = lane + 32 * i;
        if (e < E) grow[e] = c * v[i] * (f[i] - fs);
      }
    }
  }
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    const int e = lane + 32 * i;
    if (e < E) wsum[warp * E + e] = acc[i];
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    float sp = 0.f;
    for (int w = 0; w < 8; ++w) sp += wsum[w * E + e];
    part[static_cast<size_t>(blockIdx.x) * E + e] = sp;
  }
}

// P_e = (1/T) sum over blocks (block order) of the partials; f_e = counts_e / (T k);
// out = [loss, P[0..E), f[0..E)] with loss = alpha E sum_e f_e P_e (expert order).
__global__ void __launch_bounds__(1024) balance_finish_kernel(const float *__restrict__ part, int nblk, int T,
                                                              int E, int k, const int *__restrict__ counts,
                                                              float alpha, float *__restrict__ out) {
  const float inv_slots = 1.0f / (static_cast<float>(T) * static_cast<float>(k));
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    float s = 0.f;
    for (int b = 0; b < nblk; ++b) s += __ldg(part + static_cast<size_t>(b) * E + e);
    out[1 + e] = s / static_cast<float>(T);
    out[1 + E + e] = static_cast<float>(__ldg(counts + e)) * inv_slots;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float acc = 0.f;
    for (int e = 0; e < E; ++e) acc = fmaf(out[1 + E + e], out[1 + e], acc);
    out[0] = alpha * static_cast<float>(E) * acc;
  }
}

// bf16 copy of fp32 values (the router backward's dlogits operand).
__global__ void __launch_bounds__(256) to_bf16_kernel(const float *__restrict__ src, long n,
                                                      uint16_t *__restrict__ dst) {
  const long i = static_cast<long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i < n) dst[i] = static_cast<uint16_t>(pack_bf16x2(src[i], 0.f) & 0xFFFFu);  // low half = src[i]
}

// ------------------------------------------------------------ B6: reverse dispatch
__global__ void __launch_bounds__(256) reverse_dispatch_kernel(
    const uint4 *__restrict__ dX, const uint4 *__restrict__ dxs, const float *__restrict__ g, int T,
    int d, int k, int E, RouteBufs b, uint4 *__restrict__ dx, float *__restrict__ dlogits,
    const float *__restrict__ aux_grad) {
  const int t = static_cast<int>((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (t >= T) return;
  int my_row = 0, my_e = -1;
  float my_w = 0.f, my_g = 0.f;
  if (lane < k) {
    const int slot = t * k + lane;
    my_e = __ldg(b.idx + slot);
    if (MOE_BOUNDS_OK(my_e >= 0 && my_e < E, b.status)) {
      my_row = __ldg(b.poff + my_e) + __ldg(b.perm + slot) - __ldg(b.offsets + my_e);
      my_w = __ldg(b.w + slot);
      my_g = __ldg(g + slot);
      if (!MOE_BOUNDS_OK(my_row >= 0 && my_row < b.n_rows, b.status)) my_row = 0;
    } else {
      my_e = 0;
    }
  }
  // dlogits: softmax-over-k gradient w_j (g_j - sum_i w_i g_i), slot order sum.
  float S = 0.f;
  for (int j = 0; j < k; ++j)
    S = fmaf(__shfl_sync(0xffffffffu, my_w, j), __shfl_sync(0xffffffffu, my_g, j), S);
  const float dl = my_w * (my_g - S);
  // plus, with a load-balancing term, its gradient row (dense over E)
  float *drow = dlogits + static_cast<size_t>(t) * E;
  const float *arow = aux_grad ? aux_grad + static_cast<size_t>(t) * E : nullptr;
  for (int e = lane; e < E; e += 32) drow[e] = arow ? __ldg(arow + e) : 0.f;
  __syncwarp();
  if (lane < k) drow[my_e] = arow ? dl + __ldg(arow + my_e) : dl;
  const int vec = d >> 3;
  for (int i = lane; i < vec; i += 32) {
    float acc[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) acc[q] = 0.f;
    for (int j = 0; j < k; ++j) {
      const int row = __shfl_sync(0xffffffffu, my_row, j);
      float f[8];
      unpack8(__ldg(dX + static_cast<size_t>(row) * vec + i), f);
#pragma unroll
      for (int q = 0; q < 8; ++q) acc[q] += f[q];
    }
    if (dxs) {
      float f[8];
      unpack8(__ldg(dxs + static_cast<size_t>(t) * vec + i), f);
#pragma unroll
      for (int q = 0; q < 8; ++q) acc[q] += f[q];
    }
    dx[static_cast<size_t>(t) * vec + i] = pack8(acc);
  }
}

// ------------------------------------------------------------ transposes
// Block: 32 source rows x CH chunks of 256 columns, loaded up front (four
// 16-byte loads per thread and chunk) into bf16 shared-memory tiles; after one
// barrier the output rows
// (source columns) are written: for MX thread c owns output row c, one
// 32-value block, and writes its 32 codes plus the scale byte; bf16 output
// rows are written 64 bytes at a time by 4 threads each.
// ROWQ (MX, weights): the tile's source rows are also quantised along C into
// row-blocked codes rq [batch * nrows, C] with scales over K = C, so one read
// of the bf16 source gives both operand orientations.
// CANON (MX): every scale byte goes to the canonical [rows, K/32] position
// instead of the tiled operand layout (the C ABI's weight quantisers).
template <bool MX, bool GATHER, bool ROWQ = false, int CH = 1, bool CANON = false>
__global__ void __launch_bounds__(256) transpose_rows_kernel(
    const uint16_t *__restrict__ src, long src_batch_stride, int C, int nrows_host,
    const int *__restrict__ nrows_dev, long nsrc, int k, int E, RouteBufs b, void *dst,
    long dst_batch_stride, uint8_t *__restrict__ dst_sf, long sf_batch_rows, long ld_dst,
    uint8_t *__restrict__ rq = nullptr, uint8_t *__restrict__ rq_sf = nullptr) {
  __shared__ __align__(16) uint16_t tile[CH][32][256];
  const int r0 = blockIdx.x * 32;
  const int cb0 = blockIdx.y * 256 * CH;
  const int bz = blockIdx.z;
  const int nrows = nrows_dev ? __ldg(nrows_dev) : nrows_host;
  if (r0 >= nrows) return;
  src += static_cast<size_t>(bz) * src_batch_stride;
  const int tid = static_cast<int>(threadIdx.x);
  const int rr = tid >> 3;          // 0..31: source row within the block
  const int cc = (tid & 7) * 8;     // 0..56: column within a 64-column sub-tile
  const int r = r0 + rr;
  long srow = r;
  if constexpr (GATHER) srow = token_of_row(b, E, k, r, nullptr);
  const bool valid = srow >= 0 && srow < nsrc;
  int nsub[CH];
#pragma unroll
  for (int h = 0; h < CH; ++h) nsub[h] = max(0, min(4, (C - cb0 - 256 * h) / 64));
  uint4 q[CH][4];
#pragma unroll
  for (int h = 0; h < CH; ++h)
#pragma unroll
    for (int j = 0; j < 4; ++j)
      q[h][j] = (valid && j < nsub[h])
                    ? __ldg(reinterpret_cast<const uint4 *>(src + static_cast<size_t>(srow) * C + cb0 + 256 * h +
                                                            64 * j + cc))
                    : make_uint4(0, 0, 0, 0);
#pragma unroll
  for (int h = 0; h < CH; ++h) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (j >= nsub[h]) break;
      if constexpr (ROWQ) {
        float f[8];
        unpack8(q[h][j], f);
        const long qrow = static_cast<long>(bz) * nrows + r;
        const int col = cb0 + 256 * h + 64 * j + cc;
        uint32_t byte;
        const uint2 code = mx_encode8_quad(f, &byte);
        *reinterpret_cast<uint2 *>(rq + static_cast<size_t>(qrow) * C + col) = code;
        if ((tid & 3) == 0)
          rq_sf[CANON ? static_cast<size_t>(qrow) * (C / 32) + (col >> 5) : sf_tiled_offset(qrow, col >> 5, C)] =
              static_cast<uint8_t>(byte);
      }
      *reinterpret_cast<uint4 *>(&tile[h][rr][tcol(rr, 64 * j + cc)]) = q[h][j];
    }
  }
  __syncthreads();
#pragma unroll
  for (int h = 0; h < CH; ++h) {
    const int cb = cb0 + 256 * h;
    if constexpr (MX) {
      // thread c: source column cb + c = output row cb + c, one 32-value block
      if (tid < 64 * nsub[h])
        column_block_codes<CANON>(tile[h], tid, cb, r0,
                           reinterpret_cast<uint8_t *>(dst) + static_cast<size_t>(bz) * dst_batch_stride, dst_sf,
                           ld_dst, static_cast<long>(bz) * sf_batch_rows);
    } else {
      // 4 threads per output row (8 source rows each), 64 output rows per round:
      // a warp writes 8 output rows x 64 contiguous bytes per instruction
      const int c = tid >> 2, part = tid & 3;
      uint16_t *o = reinterpret_cast<uint16_t *>(dst) + static_cast<size_t>(bz) * dst_batch_stride + r0 + part * 8;
      for (int j = 0; j < nsub[h]; ++j) {
        const int col = 64 * j + c;
        uint32_t w[4];
#pragma unroll
        for (int t = 0; t < 4; ++t)
          w[t] = static_cast<uint32_t>(tile[h][part * 8 + 2 * t][tcol(part * 8 + 2 * t, col)]) |
                 (static_cast<uint32_t>(tile[h][part * 8 + 2 * t + 1][tcol(part * 8 + 2 * t + 1, col)]) << 16);
        *reinterpret_cast<uint4 *>(o + static_cast<size_t>(cb + col) * ld_dst) = make_uint4(w[0], w[1], w[2], w[3]);
      }
    }
  }
}

// Row-blocked quantisation: src [rows, cols] bf16 -> codes + scales, tiled
// (weights, GEMM operands) or canonical [rows, cols/32] (per-token codes that
// the ring dispatch gathers).
template <bool TILED>
__global__ void __launch_bounds__(256) quantize_rows_kernel(const uint4 *__restrict__ src, long rows,
                                                            int cols, uint2 *__restrict__ codes,
                                                            uint8_t *__restrict__ sf) {
  const long r = static_cast<long>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (r >= rows) return;
  const int vec = cols >> 3;
  for (int i = lane; i < vec; i += 32) {
    float f[8];
    unpack8(__ldg(src + static_cast<size_t>(r) * vec + i), f);
    uint32_t byte;
    codes[static_cast<size_t>(r) * vec + i] = mx_encode8_quad(f, &byte);
    if ((lane & 3) == 0)
      sf[TILED ? sf_tiled_offset(r, i >> 2, cols) : static_cast<size_t>(r) * (cols / 32) + (i >> 2)] =
          static_cast<uint8_t>(byte);
  }
}

// MXFP8 scales between the canonical order [rows, K/32] and the tiled operand
// layout, one 4-byte word (4 consecutive blocks of a row = 4 consecutive
// bytes in both layouts) per thread, threads in canonical order.
template <bool TO_TILED>
__global__ void __launch_bounds__(256) scales_layout_kernel(const uint32_t *__restrict__ src,
                                                            uint32_t *__restrict__ dst, long rows, int K) {
  const long kw = K / 128;  // words per row
  const long i = static_cast<long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= rows * kw) return;
  const long r = i / kw, j = i % kw;
  const size_t t = sf_tiled_offset(r, 4 * j, K) / 4;
  if (TO_TILED) dst[t] = __ldg(src + i);
  else dst[i] = __ldg(src + t);
}

// ------------------------------------------------------------ NVFP4
// Absolute maximum of each of `batch` bf16 tensors of n values (n a multiple of
// 8): blocks of grid.x stride over a tensor (grid.y), the warps' maxima are
// combined with an integer atomicMax on the fp32 bits (|v| >= 0, so the bit
// patterns order like the values; the result does not depend on the order).
// `out` must be zero beforehand.
__global__ void __launch_bounds__(256) amax_kernel(const uint4 *__restrict__ src, long n, unsigned *out) {
  const long vec = n / 8;
  const uint4 *p = src + static_cast<long>(blockIdx.y) * vec;
  float am = 0.f;
  for (long i = static_cast<long>(blockIdx.x) * blockDim.x + threadIdx.x; i < vec;
       i += static_cast<long>(gridDim.x) * blockDim.x) {
    float f[8];
    unpack8(__ldg(p + i), f);
#pragma unroll
    for (int q = 0; q < 8; ++q) am = fmaxf(am, fabsf(f[q]));
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, off));
  if ((threadIdx.x & 31) == 0) atomicMax(out + blockIdx.y, __float_as_uint(am));
}

// In place: the fp32 bits of n tensors' absolute maxima -> their NVFP4
// second-level scales 2688 / amax (1 for an all-zero tensor).
__global__ void nv_scale_from_amax_kernel(unsigned *amax_then_scale, int n) {
  const int i = static_cast<int>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i < n) amax_then_scale[i] = __float_as_uint(nv_global_scale(__uint_as_float(amax_then_scale[i])));
}

// NVFP4 rows: src [rows, cols] bf16 -> packed codes [rows, cols / 2] and scale
// codes (tiled: the GEMM operand layout, K' = 2 cols; else canonical [rows,
// cols / 16]); thread per block of 16.  Row r's tensor has the second-level
// scale gscale[r / rows_per_tensor].
template <bool TILED>
__global__ void __launch_bounds__(256) nv_quantize_rows_kernel(const uint4 *__restrict__ src, long rows, int cols,
                                                               long rows_per_tensor, const float *__restrict__ gscale,
                                                               uint2 *__restrict__ codes, uint8_t *__restrict__ sf) {
  const int nb = cols / 16;
  const long i = static_cast<long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= rows * nb) return;
  const long r = i / nb;
  const int b = static_cast<int>(i % nb);
  const float s = __ldg(gscale + r / rows_per_tensor);
  float v[16];
  unpack8(__ldg(src + 2 * i), v);
  unpack8(__ldg(src + 2 * i + 1), v + 8);
  uint32_t w[2];
  const uint32_t code = nv_block16(v, s, w);
  codes[i] = make_uint2(w[0], w[1]);
  sf[TILED ? sf_tiled_offset(r, b, 2L * cols) : static_cast<size_t>(i)] = static_cast<uint8_t>(code);
}

// NVFP4 dispatch: padded expert-sorted row pr <- the token's codes (xq [T, d/2],
// canonical scales xq_sf [T, d/16]), zeros on padding rows; scales go to the
// tiled layout of xs (K' = 2 d), 4 blocks (one word) per thread.  Warp per row.
__global__ void __launch_bounds__(256) nv_gather_kernel(const uint4 *__restrict__ xq,
                                                        const uint32_t *__restrict__ xq_sf, int d, int k, int E,
                                                        RouteBufs b, long rows, uint4 *__restrict__ xs,
                                                        uint8_t *__restrict__ xs_sf) {
  const long pr = static_cast<long>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (pr >= rows || pr >= __ldg(b.poff + E)) return;
  const int tok = token_of_row(b, E, k, static_cast<int>(pr), nullptr);
  const int vec = d / 32;  // 16-byte pieces of a row of codes
  for (int i = lane; i < vec; i += 32)
    xs[pr * vec + i] = tok >= 0 ? __ldg(xq + static_cast<long>(tok) * vec + i) : make_uint4(0, 0, 0, 0);
  const int words = d / 64;  // scale words (4 blocks of 16) of a row
  for (int j = lane; j < words; j += 32)
    *reinterpret_cast<uint32_t *>(xs_sf + sf_tiled_offset(pr, 4 * j, 2L * d)) =
        tok >= 0 ? __ldg(xq_sf + static_cast<long>(tok) * words + j) : 0u;
}

// Zeros of the empty experts' weight gradients: block (x, e) clears bytes
// [x MB, (x + 1) MB) of expert e's matrix when the expert received no rows.
constexpr long kZeroPiece = 1L << 20;

__global__ void __launch_bounds__(512) zero_empty_experts_kernel(uint8_t *__restrict__ dW, long expert_bytes,
                                                                 const int *__restrict__ counts) {
  const int e = static_cast<int>(blockIdx.y);
  if (__ldg(counts + e) != 0) return;
  const long u0 = static_cast<long>(blockIdx.x) * kZeroPiece / 16;
  const long u1 = min(u0 + kZeroPiece / 16, expert_bytes / 16);
  uint4 *p = reinterpret_cast<uint4 *>(dW + static_cast<long>(e) * expert_bytes);
  const uint4 z = make_uint4(0, 0, 0, 0);
  for (long u = u0 + threadIdx.x; u < u1; u += blockDim.x) p[u] = z;
}

inline unsigned blocks_for(long n, int per_block) {
  return static_cast<unsigned>((n + per_block - 1) / per_block);
}

}  // namespace

cudaError_t launch_route(const float *logits, int T, int E, int k, const RouteBufs &b,
                         cudaStream_t s) {
  const unsigned grid = blocks_for(T, 8);
  const int vpl = (E + 31) / 32;
  if (vpl <= 1) route_topk_kernel<1><<<grid, 256, 0, s>>>(logits, T, E, k, b.idx, b.w);
  else if (vpl <= 2) route_topk_kernel<2><<<grid, 256, 0, s>>>(logits, T, E, k, b.idx, b.w);
  else if (vpl <= 4) route_topk_kernel<4><<<grid, 256, 0, s>>>(logits, T, E, k, b.idx, b.w);
  else if (vpl <= 8) route_topk_kernel<8><<<grid, 256, 0, s>>>(logits, T, E, k, b.idx, b.w);
  else if (vpl <= 16) route_topk_kernel<16><<<grid, 256, 0, s>>>(logits, T, E, k, b.idx, b.w);
  else route_topk_kernel<32><<<grid, 256, 0, s>>>(logits, T, E, k, b.idx, b.w);
  const int R = T * k;
  const int nchunks = (R + kSchedChunk - 1) / kSchedChunk;
  const size_t smem = 4 * static_cast<size_t>(E) * sizeof(int);
  sched_hist_kernel<<<blocks_for(nchunks, 4), 128, smem, s>>>(b.idx, R, E, nchunks, b.hist, b.status);
  sched_scan_kernel<<<1, 1024, 0, s>>>(b.hist, nchunks, E, b.counts, b.offsets, b.poff);
  sched_scatter_kernel<<<blocks_for(nchunks, 4), 128, smem, s>>>(b.idx, R, E, nchunks, b.hist,
                                                                  b.offsets, b.perm, b.inv, b.status);
  return cudaGetLastError();
}

cudaError_t launch_gather(const void *x, int T, int d, int k, int E, const RouteBufs &b,
                          int64_t rp_max, bool mx, void *xs, uint8_t *xs_sf, uint8_t *xT, uint8_t *xT_sf,
                          uint8_t *xq, uint8_t *xq_sf, cudaStream_t s) {
  if (mx) {
    // Inference: every token's row codes once, then the dispatch copies them
    // per routed row.  Training reads the bf16 rows anyway (for the column-
    // blocked codes) and encodes the row codes from the same registers.
    if (xs && !xT) {
      quantize_rows_kernel<false><<<blocks_for(T, 8), 256, 0, s>>>(static_cast<const uint4 *>(x), T, d,
                                                                    reinterpret_cast<uint2 *>(xq), xq_sf);
    } else {
      xq = nullptr;
      xq_sf = nullptr;
    }
    if (b.tile_order) tile_order_kernel<<<1, kOrderBuckets, 0, s>>>(b, T, E, k, b.tile_order);
    if (xq)
      gather_mx_tile_kernel<true><<<blocks_for(rp_max, 32), 256, 0, s>>>(
          static_cast<const uint16_t *>(x), xq, xq_sf, d, k, E, b, static_cast<uint8_t *>(xs), xs_sf, xT, xT_sf,
          rp_max);
    else
      gather_mx_tile_kernel<false><<<blocks_for(rp_max, 32), 256, 0, s>>>(
          static_cast<const uint16_t *>(x), xq, xq_sf, d, k, E, b, static_cast<uint8_t *>(xs), xs_sf, xT, xT_sf,
          rp_max);
  } else
    gather_bf16_kernel<<<blocks_for(rp_max, 8), 256, 0, s>>>(static_cast<const uint4 *>(x), d, k, E, b, rp_max,
                                                              static_cast<uint4 *>(xs));
  return cudaGetLastError();
}

cudaError_t launch_zero_empty_experts(void *dW, int E, long expert_bytes, const int *counts, cudaStream_t s) {
  if (!dW || !counts || E <= 0 || E > 65535 || expert_bytes <= 0 || expert_bytes % 16 != 0 ||
      reinterpret_cast<uintptr_t>(dW) % 16 != 0)
    return cudaErrorInvalidValue;
  const dim3 grid(static_cast<unsigned>((expert_bytes + kZeroPiece - 1) / kZeroPiece), static_cast<unsigned>(E));
  zero_empty_experts_kernel<<<grid, 512, 0, s>>>(static_cast<uint8_t *>(dW), expert_bytes, counts);
  return cudaGetLastError();
}

cudaError_t launch_combine(const void *o, const void *s_out, int T, int d, int k, int E,
                           const RouteBufs &b, void *y, cudaStream_t s) {
  combine_kernel<<<blocks_for(T, 8), 256, 0, s>>>(static_cast<const uint4 *>(o),
                                                  static_cast<const uint4 *>(s_out), T, d, k, E, b,
                                                  static_cast<uint4 *>(y));
  return cudaGetLastError();
}

cudaError_t launch_reverse_combine(const void *dy, const void *o, int T, int d, int k, int E,
                                   const RouteBufs &b, int64_t rp_max, void *dO, float *g, cudaStream_t s) {
  (void)T;
  reverse_combine_kernel<<<blocks_for(rp_max, 8), 256, 0, s>>>(static_cast<const uint4 *>(dy),
                                                               static_cast<const uint4 *>(o), d, k, E, b, rp_max,
                                                               static_cast<uint4 *>(dO), g);
  return cudaGetLastError();
}

cudaError_t launch_reverse_combine_mx(const void *dy, const void *o, int T, int d, int k, int E,
                                      const RouteBufs &b, int64_t rp_max, float *g, uint8_t *dOq,
                                      uint8_t *dOq_sf, uint8_t *dOT, uint8_t *dOT_sf, cudaStream_t s) {
  if (b.tile_order) tile_order_kernel<<<1, kOrderBuckets, 0, s>>>(b, T, E, k, b.tile_order);
  reverse_combine_mx_kernel<<<blocks_for(rp_max, 32), 256, 0, s>>>(
      static_cast<const uint16_t *>(dy), static_cast<const uint16_t *>(o), d, k, E, b, g, dOq, dOq_sf,
      dOT, dOT_sf, rp_max);
  return cudaGetLastError();
}

cudaError_t launch_reverse_dispatch(const void *dX, const void *dxs, const float *g, int T,
                                    int d, int k, int E, const RouteBufs &b, void *dx,
                                    float *dlogits, const float *aux_grad, cudaStream_t s) {
  reverse_dispatch_kernel<<<blocks_for(T, 8), 256, 0, s>>>(
      static_cast<const uint4 *>(dX), static_cast<const uint4 *>(dxs), g, T, d, k, E, b,
      static_cast<uint4 *>(dx), dlogits, aux_grad);
  return cudaGetLastError();
}

cudaError_t launch_transpose_rows(const void *src, int C, int nrows_out, const int *nrows_dev,
                                  long nsrc, bool gather, int k, int E, const RouteBufs *b,
                                  int64_t rows_alloc, void *dst, int64_t ld_dst, cudaStream_t s) {
  const dim3 grid(blocks_for(rows_alloc, 32), blocks_for(C, 256), 1);
  const RouteBufs bb = b ? *b : RouteBufs{};
  const uint16_t *sp = static_cast<const uint16_t *>(src);
  const long ns = gather ? (1L << 40) : nsrc;
  if (gather)
    transpose_rows_kernel<false, true><<<grid, 256, 0, s>>>(sp, 0, C, nrows_out, nrows_dev, ns, k, E, bb, dst,
                                                            0, nullptr, 0, ld_dst);
  else
    transpose_rows_kernel<false, false><<<grid, 256, 0, s>>>(sp, 0, C, nrows_out, nrows_dev, ns, k, E, bb, dst,
                                                             0, nullptr, 0, ld_dst);
  return cudaGetLastError();
}

cudaError_t launch_quantize_mx(const void *src, int batch, int rows, int cols, bool transpose,
                               uint8_t *codes, uint8_t *scales, bool canon, cudaStream_t s) {
  if (!transpose) {
    const long total = static_cast<long>(batch) * rows;
    if (canon)
      quantize_rows_kernel<false><<<blocks_for(total, 8), 256, 0, s>>>(
          static_cast<const uint4 *>(src), total, cols, reinterpret_cast<uint2 *>(codes), scales);
    else
      quantize_rows_kernel<true><<<blocks_for(total, 8), 256, 0, s>>>(
          static_cast<const uint4 *>(src), total, cols, reinterpret_cast<uint2 *>(codes), scales);
  } else {
    const dim3 grid(blocks_for(rows, 32), blocks_for(cols, 256), batch);
#define MOE_QT(CANON)                                                                                       \
  transpose_rows_kernel<true, false, false, 1, CANON><<<grid, 256, 0, s>>>(                                  \
      static_cast<const uint16_t *>(src), static_cast<long>(rows) * cols, cols, rows, nullptr, rows, 1, 1, \
      RouteBufs{}, codes, static_cast<long>(rows) * cols, scales, cols, rows)
    if (canon) MOE_QT(true);
    else MOE_QT(false);
#undef MOE_QT
  }
  return cudaGetLastError();
}

int balance_blocks(int T) { return static_cast<int>((T + kBalanceTokensPerBlock - 1) / kBalanceTokensPerBlock); }

cudaError_t launch_balance(const float *logits, int T, int E, int k, const int *counts, float alpha, float *part,
                           float *grad, float *out, cudaStream_t s) {
  const int nblk = balance_blocks(T);
  const int vpl = (E + 31) / 32;
  const size_t smem = 8 * static_cast<size_t>(E) * sizeof(float);
#define MOE_BAL(V) \
  balance_kernel<V><<<nblk, 256, smem, s>>>(logits, T, E, k, counts, alpha, kBalanceTokensPerBlock, part, grad)
  if (vpl <= 1) MOE_BAL(1);
  else if (vpl <= 2) MOE_BAL(2);
  else if (vpl <= 4) MOE_BAL(4);
  else if (vpl <= 8) MOE_BAL(8);
  else if (vpl <= 16) MOE_BAL(16);
  else MOE_BAL(32);
#undef MOE_BAL
  balance_finish_kernel<<<1, 1024, 0, s>>>(part, nblk, T, E, k, counts, alpha, out);
  return cudaGetLastError();
}

// Thread per 8 output columns of one row (one 16-byte store).
__global__ void __launch_bounds__(256) pad_to_bf16_kernel(const float *__restrict__ src, int rows, int cols,
                                                          int rows_p, int cols_p, uint4 *__restrict__ dst) {
  const long i = static_cast<long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int per_row = cols_p / 8;
  if (i >= static_cast<long>(rows_p) * per_row) return;
  const int r = static_cast<int>(i / per_row);
  const int c0 = static_cast<int>(i % per_row) * 8;
  float f[8];
#pragma unroll
  for (int q = 0; q < 8; ++q)
    f[q] = (r < rows && c0 + q < cols) ? __ldg(src + static_cast<size_t>(r) * cols + c0 + q) : 0.f;
  dst[i] = pack8(f);
}

__global__ void __launch_bounds__(256) crop_f32_kernel(const float *__restrict__ src, int rows, int cols,
                                                       long ld_src, float *__restrict__ dst) {
  const long i = static_cast<long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= static_cast<long>(rows) * cols) return;
  const long r = i / cols, c = i % cols;
  dst[i] = __ldg(src + r * ld_src + c);
}

cudaError_t launch_pad_to_bf16(const float *src, int rows, int cols, int rows_p, int cols_p, void *dst,
                               cudaStream_t s) {
  const long n = static_cast<long>(rows_p) * (cols_p / 8);
  pad_to_bf16_kernel<<<blocks_for(n, 256), 256, 0, s>>>(src, rows, cols, rows_p, cols_p, static_cast<uint4 *>(dst));
  return cudaGetLastError();
}

cudaError_t launch_crop_f32(const float *src, int rows, int cols, long ld_src, float *dst, cudaStream_t s) {
  crop_f32_kernel<<<blocks_for(static_cast<long>(rows) * cols, 256), 256, 0, s>>>(src, rows, cols, ld_src, dst);
  return cudaGetLastError();
}

cudaError_t launch_to_bf16(const float *src, long n, void *dst, cudaStream_t s) {
  to_bf16_kernel<<<blocks_for(n, 256), 256, 0, s>>>(src, n, static_cast<uint16_t *>(dst));
  return cudaGetLastError();
}

cudaError_t launch_quantize_mx_both(const void *src, int batch, int rows, int cols, uint8_t *codes,
                                    uint8_t *scales, uint8_t *codes_t, uint8_t *scales_t, bool canon,
                                    cudaStream_t s) {
  // two 256-column chunks per block (twice the loads in flight) when they tile cols
#define MOE_QB(CH, CANON)                                                                                    \
  transpose_rows_kernel<true, false, true, CH, CANON><<<grid, 256, 0, s>>>(                                  \
      static_cast<const uint16_t *>(src), static_cast<long>(rows) * cols, cols, rows, nullptr, rows, 1, 1,  \
      RouteBufs{}, codes_t, static_cast<long>(rows) * cols, scales_t, cols, rows, codes, scales)
  if (cols % 512 == 0) {
    const dim3 grid(blocks_for(rows, 32), blocks_for(cols, 512), batch);
    if (canon) MOE_QB(2, true);
    else MOE_QB(2, false);
  } else {
    const dim3 grid(blocks_for(rows, 32), blocks_for(cols, 256), batch);
    if (canon) MOE_QB(1, true);
    else MOE_QB(1, false);
  }
#undef MOE_QB
  return cudaGetLastError();
}

cudaError_t launch_scales_layout(const void *src, long rows, int K, bool to_tiled, void *dst, cudaStream_t s) {
  const long n = rows * (K / 128);
  if (to_tiled)
    scales_layout_kernel<true><<<blocks_for(n, 256), 256, 0, s>>>(static_cast<const uint32_t *>(src),
                                                                   static_cast<uint32_t *>(dst), rows, K);
  else
    scales_layout_kernel<false><<<blocks_for(n, 256), 256, 0, s>>>(static_cast<const uint32_t *>(src),
                                                                    static_cast<uint32_t *>(dst), rows, K);
  return cudaGetLastError();
}

cudaError_t launch_nv_global_scales(const void *src, int batch, long n, float *gscale, cudaStream_t s) {
  unsigned *g = reinterpret_cast<unsigned *>(gscale);
  const cudaError_t e = cudaMemsetAsync(g, 0, static_cast<size_t>(batch) * sizeof(unsigned), s);
  if (e != cudaSuccess) return e;
  long blocks = (n / 8 + 255) / 256;
  if (blocks > 1024) blocks = 1024;
  amax_kernel<<<dim3(static_cast<unsigned>(blocks), batch), 256, 0, s>>>(static_cast<const uint4 *>(src), n, g);
  nv_scale_from_amax_kernel<<<blocks_for(batch, 256), 256, 0, s>>>(g, batch);
  return cudaGetLastError();
}

cudaError_t launch_nv_quantize_rows(const void *src, long rows, int cols, long rows_per_tensor, const float *gscale,
                                    uint8_t *codes, uint8_t *scales, bool tiled, cudaStream_t s) {
  const long n = rows * (cols / 16);
  if (tiled)
    nv_quantize_rows_kernel<true><<<blocks_for(n, 256), 256, 0, s>>>(
        static_cast<const uint4 *>(src), rows, cols, rows_per_tensor, gscale, reinterpret_cast<uint2 *>(codes),
        scales);
  else
    nv_quantize_rows_kernel<false><<<blocks_for(n, 256), 256, 0, s>>>(
        static_cast<const uint4 *>(src), rows, cols, rows_per_tensor, gscale, reinterpret_cast<uint2 *>(codes),
        scales);
  return cudaGetLastError();
}

cudaError_t launch_nv_gather(const uint8_t *xq, const uint8_t *xq_sf, int d, int k, int E, const RouteBufs &b,
                             long rows, uint8_t *xs, uint8_t *xs_sf, cudaStream_t s) {
  nv_gather_kernel<<<blocks_for(rows, 8), 256, 0, s>>>(reinterpret_cast<const uint4 *>(xq),
                                                       reinterpret_cast<const uint32_t *>(xq_sf), d, k, E, b, rows,
                                                       reinterpret_cast<uint4 *>(xs), xs_sf);
  return cudaGetLastError();
}

cudaError_t launch_quantize_tokens(const void *x, int T, int d, uint8_t *codes, uint8_t *scales,
                                   cudaStream_t s) {
  quantize_rows_kernel<false><<<blocks_for(T, 8), 256, 0, s>>>(static_cast<const uint4 *>(x), T, d,
                                                                reinterpret_cast<uint2 *>(codes), scales);
  return cudaGetLastError();
}

cudaError_t launch_transpose_bf16(const void *src, int batch, int rows, int cols, void *dst,
                                  cudaStream_t s) {
  const dim3 grid(blocks_for(rows, 32), blocks_for(cols, 256), batch);
  transpose_rows_kernel<false, false><<<grid, 256, 0, s>>>(
      static_cast<const uint16_t *>(src), static_cast<long>(rows) * cols, cols, rows, nullptr, rows, 1,
      1, RouteBufs{}, dst, static_cast<long>(rows) * cols, nullptr, 0, rows);
  return cudaGetLastError();
}

}  // namespace moe
