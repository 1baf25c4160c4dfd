// Dispatch helpers shared by the stand-alone dispatch kernel and the gather
// CTAs of the persistent ring kernel: bf16 unpacking, 4-lane MXFP8 block
// encoding, the token of an expert-sorted row, and the 32-row dispatch tile.
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
  const int slot = __ldg(b.inv + __ldg(b.offsets + e) + local);
  if (slot_out) *slot_out = slot;
  return slot / k;
}

// MXFP8 dispatch of the 32 expert-sorted padded rows [r0, r0 + 32) by 256
// threads: each row's token is read from x [T, d] (bf16, zeros for padding
// rows) and, unless dst is NULL, quantised along d into codes at dst row
// q0 + i (row stride d) with tiled scales (K = d).  When xT is given, the
// same 32 rows are also quantised per column (one 32-row block) into the
// transposed codes xT [d, ld_t] at columns r0 .. r0 + 31, with tiled scales
// (K = ld_t).  `tile` is 32 x 65 floats of shared memory; `sync()` is a
// barrier over the 256 threads.
template <typename Sync>
MOE_DEV void dispatch_rows32(const uint16_t *__restrict__ x, int d, int k, int E, const RouteBufs &b, int r0,
                             int q0, uint8_t *__restrict__ dst, uint8_t *__restrict__ dst_sf,
                             uint8_t *__restrict__ xT, uint8_t *__restrict__ xT_sf, long ld_t,
                             float (*tile)[65], int tid, Sync sync) {
  const int rr = tid >> 3;
  const int cc = (tid & 7) * 8;
  const int pr = r0 + rr;
  const int qr = q0 + rr;
  const int tok = token_of_row(b, E, k, pr, nullptr);
  const uint16_t *xr = x + static_cast<size_t>(tok < 0 ? 0 : tok) * d;
  const int c = tid >> 2;
  const int part = tid & 3;
  for (int cb = 0; cb < d; cb += 256) {
    uint4 q[4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
      q[j] = tok >= 0 ? __ldg(reinterpret_cast<const uint4 *>(xr + cb + 64 * j + cc)) : make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      float f[8];
      unpack8(q[j], f);
      if (dst) {
        const int col = cb + 64 * j + cc;
        uint32_t byte;
        const uint2 code = mx_encode8_quad(f, &byte);
        *reinterpret_cast<uint2 *>(dst + static_cast<size_t>(qr) * d + col) = code;
        if ((tid & 3) == 0) dst_sf[sf_tiled_offset(qr, col >> 5, d)] = static_cast<uint8_t>(byte);
      }
      if (xT) {
        sync();
#pragma unroll
        for (int t = 0; t < 8; ++t) tile[rr][cc + t] = f[t];
        sync();
        float v[8];
#pragma unroll
        for (int t = 0; t < 8; ++t) v[t] = tile[part * 8 + t][c];
        const size_t ocol = static_cast<size_t>(cb + 64 * j + c);
        uint32_t tb;
        const uint2 tcode = mx_encode8_quad(v, &tb);
        *reinterpret_cast<uint2 *>(xT + ocol * ld_t + r0 + part * 8) = tcode;
        if (part == 0) xT_sf[sf_tiled_offset(static_cast<long>(ocol), r0 / 32, ld_t)] = static_cast<uint8_t>(tb);
      }
    }
  }
}

}  // namespace moe
