// Dispatch helpers: bf16 unpacking, 4-lane MXFP8 block encoding, the token of
// an expert-sorted row (also used by the gather CTAs of the persistent ring
// kernel), column-blocked codes of a 32-row tile, and the 32-row dispatch tile.
//
// Method reference ("Mixture-of-Kittens" wiki page, Key claims, MXFP8 bullet):
// activations are quantised to MXFP8 inside the dispatch.
#pragma once

#include "common.cuh"
#include "kernels.h"

namespace moe {

MOE_DEV void unpack8(const uint4 &q, float *f) {
  f[0] = bf16lo(q.x); f[1] = bf16hi(q.x);
  f[2] = bf16lo(q.y); f[3] = bf16hi(q.y);
  f[4] = bf16lo(q.z); f[5] = bf16hi(q.z);
  f[6] = bf16lo(q.w); f[7] = bf16hi(q.w);
}
MOE_DEV uint4 pack8(const float *f) {
  return make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                    pack_bf16x2(f[6], f[7]));
}
// MX-encode 8 values owned by this lane; the 4 lanes (lane & ~3 .. +3) hold one
// 32-element block.  Returns the 8 codes; *byte gets the block's scale byte.
MOE_DEV uint2 mx_encode8_quad(const float *f, uint32_t *byte) {
  float am = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) am = fmaxf(am, fabsf(f[i]));
  am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 1));
  am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 2));
  const uint32_t b = mx_scale_byte(am);
  const float s = mx_inv_scale(b);
  uint2 c;
  c.x = e4m3x2(f[0] * s, f[1] * s) | (e4m3x2(f[2] * s, f[3] * s) << 16);
  c.y = e4m3x2(f[4] * s, f[5] * s) | (e4m3x2(f[6] * s, f[7] * s) << 16);
  *byte = b;
  return c;
}

// Token of padded expert-sorted row pr, or -1 for a padding row.
MOE_DEV int token_of_row(const RouteBufs &b, int E, int k, int pr, int *slot_out) {
  const int e = expert_of_row(b.poff, E, pr);
  const int local = pr - __ldg(b.poff + e);
  if (local >= __ldg(b.counts + e)) return -1;
  if (!MOE_BOUNDS_OK(local >= 0 && __ldg(b.offsets + e) + local < b.n_slots, b.status)) return -1;
  const int slot = __ldg(b.inv + __ldg(b.offsets + e) + local);
  if (!MOE_BOUNDS_OK(slot >= 0 && slot < b.n_slots && slot / k < b.n_tok, b.status)) return -1;
  if (slot_out) *slot_out = slot;
  return slot / k;
}

// Column of element (r, c) in a 32 x 256 bf16 shared-memory tile: the 16-byte
// chunks of rows 8 apart are swizzled (chunk index XOR (r / 8) % 4), so that
// four threads reading one column at rows 0, 8, 16, 24 hit different banks,
// while a row's aligned 128-byte runs stay contiguous for 16-byte writes.
MOE_DEV int tcol(int r, int c) { return (((c >> 3) ^ ((r >> 3) & 3)) << 3) | (c & 7); }

// Column-blocked MXFP8 codes of one 256-column chunk of a 32-row tile held in
// shared memory as bf16 (tile[row][tcol(row, col)]): thread c (of
// 256) owns column c, i.e. one 32-value block, and writes its 32 codes to row
// col0 + c of the transposed codes (row stride ld_t) at columns r0 .. r0 + 31,
// and the block's scale byte into the tiled scales (K = ld_t) at row
// sf_row0 + col0 + c.
template <bool CANON = false>
MOE_DEV void column_block_codes(const uint16_t (*tile)[256], int c, long col0, int r0, uint8_t *__restrict__ dT,
                                uint8_t *__restrict__ dT_sf, long ld_t, long sf_row0 = 0) {
  float v[32];
  float am = 0.f;
#pragma unroll
  for (int r = 0; r < 32; ++r) {
    v[r] = __uint_as_float(static_cast<uint32_t>(tile[r][tcol(r, c)]) << 16);
    am = fmaxf(am, fabsf(v[r]));
  }
  const uint32_t byte = mx_scale_byte(am);
  uint32_t w[8];
  mx_encode32(v, byte, w);
  const long ocol = col0 + c;
  st_global_32B(dT + ocol * ld_t + r0, w);
  const long srow = sf_row0 + ocol;
  dT_sf[CANON ? static_cast<size_t>(srow) * (ld_t / 32) + r0 / 32 : sf_tiled_offset(srow, r0 / 32, ld_t)] =
      static_cast<uint8_t>(byte);
}

// MXFP8 dispatch of the 32 expert-sorted padded rows [r0, r0 + 32) by 256
// threads.  Unless dst is NULL, the row-blocked codes (blocks of 32 along d)
// of each row's token go to dst rows r0 .. r0 + 31 (row stride d) with tiled
// scales (K = d), zeros for padding rows: with xq given they are copied from
// the codes every token got once beforehand (xq [T, d], canonical scales
// xq_sf [T, d / 32]); otherwise they are encoded here from x [T, d] (bf16).
// When xT is given, the same 32 rows of x are also quantised per column (one
// 32-row block) into the transposed codes xT [d, ld_t] at columns r0 .. r0 +
// 31, with tiled scales (K = ld_t), through `tile` (two 32 x 256 bf16 buffers,
// one barrier per 256-column chunk).  Columns are swept 256 at a time with the
// next chunk's loads in flight.  COPY: xq is given, dst is not NULL and xT is
// NULL (inference).
template <bool COPY>
MOE_DEV void dispatch_rows32(const uint16_t *__restrict__ x, const uint8_t *__restrict__ xq,
                             const uint8_t *__restrict__ xq_sf, int d, int k, int E, const RouteBufs &b, int r0,
                             uint8_t *__restrict__ dst, uint8_t *__restrict__ dst_sf, uint8_t *__restrict__ xT,
                             uint8_t *__restrict__ xT_sf, long ld_t, uint16_t (*tile)[32][256], int tid) {
  constexpr bool copy = COPY;    // row codes copied from the per-token codes
  constexpr bool need_x = !COPY;  // bf16 rows read (row encode and/or column codes)
  const int rr = tid >> 3;                // row of this thread's loads
  const int c8 = tid & 7;
  const int pr = r0 + rr;
  const int tok = token_of_row(b, E, k, pr, nullptr);
  const uint16_t *xr = x + static_cast<size_t>(tok < 0 ? 0 : tok) * d;
  const uint8_t *qr = COPY ? xq + static_cast<size_t>(tok < 0 ? 0 : tok) * d : nullptr;
  // scales (copy): threads 0..63 move one 4-byte group (4 blocks of 32) of row tid / 2
  const int srow = tid >> 1;
  const int stok = (copy && tid < 64) ? token_of_row(b, E, k, r0 + srow, nullptr) : -1;
  auto load = [&](int cb, uint4 *q, uint4 *c, uint32_t *sw) {
    const bool in = cb < d;
    if constexpr (need_x) {
#pragma unroll
      for (int j = 0; j < 4; ++j)
        q[j] = (in && tok >= 0) ? __ldg(reinterpret_cast<const uint4 *>(xr + cb + 64 * j + 8 * c8))
                                : make_uint4(0, 0, 0, 0);
    }
    if constexpr (COPY) {
#pragma unroll
      for (int j = 0; j < 2; ++j)
        c[j] = (in && tok >= 0) ? __ldg(reinterpret_cast<const uint4 *>(qr + cb + 128 * j + 16 * c8))
                                : make_uint4(0, 0, 0, 0);
      *sw = (in && tid < 64 && stok >= 0)
                ? __ldg(reinterpret_cast<const uint32_t *>(xq_sf + static_cast<size_t>(stok) * (d / 32) + cb / 32 +
                                                            4 * (tid & 1)))
                : 0u;
    }
  };
  uint4 q[4], c[2], qn[4], cn[2];
  uint32_t sw = 0u, swn = 0u;
  load(0, q, c, &sw);
  int buf = 0;
  for (int cb = 0; cb < d; cb += 256) {
    load(cb + 256, qn, cn, &swn);  // the next chunk's loads in flight while this one is written
    if constexpr (COPY) {
#pragma unroll
      for (int j = 0; j < 2; ++j)
        *reinterpret_cast<uint4 *>(dst + static_cast<size_t>(pr) * d + cb + 128 * j + 16 * c8) = c[j];
      if (tid < 64)
        *reinterpret_cast<uint32_t *>(dst_sf + sf_tiled_offset(r0 + srow, cb / 32 + 4 * (tid & 1), d)) = sw;
    } else if (dst) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int col = cb + 64 * j + 8 * c8;
        float f[8];
        unpack8(q[j], f);
        uint32_t byte;
        const uint2 code = mx_encode8_quad(f, &byte);  // the 4 threads of a 32-column block
        *reinterpret_cast<uint2 *>(dst + static_cast<size_t>(pr) * d + col) = code;
        if ((tid & 3) == 0) dst_sf[sf_tiled_offset(pr, col >> 5, d)] = static_cast<uint8_t>(byte);
      }
    }
    if (!COPY && xT) {
#pragma unroll
      for (int j = 0; j < 4; ++j) *reinterpret_cast<uint4 *>(&tile[buf][rr][tcol(rr, 64 * j + 8 * c8)]) = q[j];
      __syncthreads();
      column_block_codes(tile[buf], tid, cb, r0, xT, xT_sf, ld_t);
      buf ^= 1;
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) q[j] = qn[j];
    c[0] = cn[0];
    c[1] = cn[1];
    sw = swn;
  }
}

}  // namespace moe
