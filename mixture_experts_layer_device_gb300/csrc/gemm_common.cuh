// Epilogue helpers shared by the 1-CTA and 2-CTA grouped GEMM kernels.
#pragma once

#include "common.cuh"
#include "kernels.h"

namespace moe {

// Per-device memo of a launch-configuration query (the answer depends only on
// the kernel and the device): the query runs once per device, outside any
// stream capture that follows.  0 means "not known yet" (answers are >= 1).
template <typename F>
inline int per_device_memo(int (&slot)[64], F query) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return query();
  if (slot[dev] <= 0) slot[dev] = query();
  return slot[dev];
}

namespace gemm_detail {

MOE_DEV void load_bf16x32(const void *base, long row, long ld, long col, float *v) {
  const uint4 *src =
      reinterpret_cast<const uint4 *>(reinterpret_cast<const __nv_bfloat16 *>(base) + row * ld + col);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint4 q = src[i];
    v[8 * i + 0] = bf16lo(q.x); v[8 * i + 1] = bf16hi(q.x);
    v[8 * i + 2] = bf16lo(q.y); v[8 * i + 3] = bf16hi(q.y);
    v[8 * i + 4] = bf16lo(q.z); v[8 * i + 5] = bf16hi(q.z);
    v[8 * i + 6] = bf16lo(q.w); v[8 * i + 7] = bf16hi(q.w);
  }
}

// 32 floats -> 16 words of bf16 pairs (round to nearest even).
MOE_DEV void bf16x32_words(const float *v, uint32_t *w) {
#pragma unroll
  for (int i = 0; i < 16; ++i) w[i] = pack_bf16x2(v[2 * i], v[2 * i + 1]);
}

// MX block of 32 values owned by this thread -> 8 code words; returns the scale byte.
MOE_DEV uint32_t mx_block_words(const float *v, uint32_t *w) {
  float am = 0.f;
#pragma unroll
  for (int i = 0; i < 32; ++i) am = fmaxf(am, fabsf(v[i]));
  const uint32_t byte = mx_scale_byte(am);
  mx_encode32(v, byte, w);
  return byte;
}

// One epilogue output: base pointer, row stride (bytes), rows that exist,
// element size.
struct OutView {
  uint8_t *p;
  long ld;
  long rows;
  int esz;
};

MOE_DEV OutView out_view(void *p, long ld_elems, long rows, int esz) {
  return OutView{static_cast<uint8_t *>(p), ld_elems * esz, rows, esz};
}

// Per-warp writer of 32-row x 64-byte output pieces: each lane places its row's
// 64 bytes in a 64-byte-swizzled shared-memory buffer (conflict-free); the
// warp reads the piece back transposed, 8 rows x 64 bytes per instruction, and
// writes it with coalesced 16-byte global stores.  The buffer is free again as
// soon as the read-back is done, so a multi-piece epilogue never waits for an
// earlier store, and the stores do not queue behind the producer's TMA loads.
struct Stager {
  uint8_t *buf;  // 2 KB, 16-byte aligned
  MOE_DEV explicit Stager(uint8_t *b) : buf(b) {}
  MOE_DEV void put(const OutView &o, const uint32_t *w16, int c0, int row0, int lane) {
    __syncwarp();  // every lane has read back the previous piece
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int jj = j ^ ((lane >> 1) & 3);
      *reinterpret_cast<uint4 *>(buf + lane * 64 + jj * 16) =
          make_uint4(w16[4 * j], w16[4 * j + 1], w16[4 * j + 2], w16[4 * j + 3]);
    }
    __syncwarp();
    // Lane (j = lane % 4, rr = lane / 4) moves 16-byte chunk j of rows rr,
    // rr + 8, rr + 16, rr + 24.  The swizzle term (row / 2) % 4 is the same for
    // the four rows, so the shared-memory reads are one base plus 512 i, and
    // the global rows one pointer plus 8 i rows.
    const int j = lane & 3;
    const int rr = lane >> 2;
    const uint8_t *src = buf + rr * 64 + ((j ^ ((rr >> 1) & 3)) * 16);
    uint8_t *dst = o.p + static_cast<long>(c0) * o.esz + j * 16 + (static_cast<long>(row0) + rr) * o.ld;
    const long step = 8 * o.ld;
    if (static_cast<long>(row0) + 32 <= o.rows) {
#pragma unroll
      for (int i = 0; i < 4; ++i)
        *reinterpret_cast<uint4 *>(dst + i * step) = *reinterpret_cast<const uint4 *>(src + 512 * i);
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i)
        if (static_cast<long>(row0) + rr + 8 * i < o.rows)
          *reinterpret_cast<uint4 *>(dst + i * step) = *reinterpret_cast<const uint4 *>(src + 512 * i);
    }
  }
  MOE_DEV void put_bf16(const OutView &o, const float *v32, int c0, int row0, int lane) {
    uint32_t w[16];
    bf16x32_words(v32, w);
    put(o, w, c0, row0, lane);
  }
  // Column-blocked MXFP8 codes of a 32 x 32 piece: each lane's 32 values (its
  // row, columns c0 .. c0 + 31) are rounded to bf16 and staged; lane c then
  // reads column c0 + c over the 32 rows (one 32-row block, rows row0 ..
  // row0 + 31) and writes its 32 codes to row c0 + c of dT (row stride ldT)
  // and the scale byte to the tiled scales dT_sf (K = ldT).
  MOE_DEV void put_col_codes(const float *v32, uint8_t *dT, uint8_t *dT_sf, long ldT, int c0, int row0,
                             int lane) {
    uint32_t w[16];
    bf16x32_words(v32, w);
    __syncwarp();
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int jj = j ^ ((lane >> 1) & 3);
      *reinterpret_cast<uint4 *>(buf + lane * 64 + jj * 16) =
          make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
    }
    __syncwarp();
    // Row r's chunk for this lane's column is (lane / 8) XOR ((r / 2) % 4): four
    // per-lane bases, one per value of (r / 2) % 4, plus r * 64 (an immediate).
    const uint8_t *base[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) base[c] = buf + (((lane >> 3) ^ c) * 16) + (lane & 7) * 2;
    float v[32];
    float am = 0.f;
#pragma unroll
    for (int r = 0; r < 32; ++r) {
      const uint16_t b = *reinterpret_cast<const uint16_t *>(base[(r >> 1) & 3] + r * 64);
      v[r] = __uint_as_float(static_cast<uint32_t>(b) << 16);
      am = fmaxf(am, fabsf(v[r]));
    }
    const uint32_t byte = mx_scale_byte(am);
    uint32_t cw[8];
    mx_encode32(v, byte, cw);
    const long orow = static_cast<long>(c0) + lane;
    st_global_32B(dT + orow * ldT + row0, cw);
    dT_sf[sf_tiled_offset(orow, row0 / 32, ldT)] = static_cast<uint8_t>(byte);
  }
};

// Four NVFP4 blocks (64 values) of one row, second-level scale 1 -> 32 bytes of
// packed codes (one 32-byte store, the lane's own row) + 4 scale bytes (next to
// each other in one 512-byte atom of the NVFP4 layout: K' = 2 ldq).
MOE_DEV void put_nv64(const GemmArgs &g, const float *v64, int col, long grow) {
  if (grow >= g.out_rows) return;
  uint32_t w[8];
  uint32_t sfw = 0;
#pragma unroll
  for (int b = 0; b < 4; ++b) sfw |= nv_block16(v64 + 16 * b, 1.0f, w + 2 * b) << (8 * b);
  st_global_32B(g.outq + grow * (g.ldq / 2) + col / 2, w);
  *reinterpret_cast<uint32_t *>(g.outq_sf + sf_tiled_offset(grow, col / 16, 2 * g.ldq)) = sfw;
}

// Two MX blocks (64 values) of one row -> one 64-byte codes piece + 2 scale bytes.
MOE_DEV void put_mx64(Stager &st, const OutView &vq, uint8_t *sf, long ldq, const float *v64,
                      int col, int row0, long grow, int lane) {
  uint32_t w[16];
  const uint32_t b0 = mx_block_words(v64, w);
  const uint32_t b1 = mx_block_words(v64 + 32, w + 8);
  st.put(vq, w, col, row0, lane);
  // (col / 32) is even, so both bytes sit next to each other in one 512-byte atom.
  *reinterpret_cast<uint16_t *>(sf + sf_tiled_offset(grow, col / 32, ldq)) =
      static_cast<uint16_t>(b0 | (b1 << 8));
}


// Drains one tile's accumulator (this warp's 32 TMEM lanes at `tb`) and writes
// the epilogue's outputs through the stager.  `release()` is called once the last
// accumulator column has been read (the MMA may then reuse it).  With
// store == false the accumulator is drained and released but nothing is
// written (the idle half of a 2-CTA tile).
template <int EPI, int BN, typename Release>
MOE_DEV void epilogue_tile(const GemmArgs &g, const OutView &vO, const OutView &vO2,
                           const OutView &vQ, Stager &st, uint32_t tb, int nk, int row0,
                           long grow, int out_col, int lane, bool store, Release release) {
  if constexpr (EPI == EPI_STORE) {
    constexpr int NCH = BN / 64;
    if (nk == 0) {  // empty reduction (an expert with no rows): zeros
      release();
      if (store) {
        float z[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) z[i] = 0.f;
#pragma unroll 1
        for (int c = 0; c < 2 * NCH; ++c) st.put_bf16(vO, z, out_col + 32 * c, row0, lane);
      }
      return;
    }
    // The whole row is drained into registers as packed bf16 pairs (TMEM loads
    // of 32 columns ping-pong with the conversion), TMEM is released, and only
    // then are the pieces staged and stored: the accumulator is never held
    // while the stores drain.
    constexpr int NC32 = BN / 32;
    uint32_t pk[BN / 2];
    uint32_t buf[2][32];
    tmem_ld32_async(tb, buf[0]);
    tmem_ld_wait();
    reg_fence<32>(buf[0]);
#pragma unroll
    for (int c = 0; c < NC32; ++c) {
      if (c + 1 < NC32) tmem_ld32_async(tb + 32 * (c + 1), buf[(c + 1) & 1]);
      bf16x32_words(reinterpret_cast<const float *>(buf[c & 1]), pk + 16 * c);
      if (c + 1 < NC32) {
        tmem_ld_wait();
        reg_fence<32>(buf[(c + 1) & 1]);
      }
    }
    release();
    if (store) {
#pragma unroll
      for (int c = 0; c < NC32; ++c) st.put(vO, pk + 16 * c, out_col + 32 * c, row0, lane);
    }
  } else if constexpr (EPI == EPI_SWIGLU) {
    // accumulator columns [0,128) = gate G, [128,256) = up U of 128 h columns
    if (!g.out && !g.out2 && g.outq) {
      // Inference with MXFP8 h: compute the 128 codes of this row (4 blocks)
      // while reading TMEM, release it, then store.
      uint32_t cw[32];
      uint32_t sb[4];
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t gr[64], ur[64];
        tmem_ld32_async(tb + 64 * c, gr);
        tmem_ld32_async(tb + 64 * c + 32, gr + 32);
        tmem_ld32_async(tb + 128 + 64 * c, ur);
        tmem_ld32_async(tb + 128 + 64 * c + 32, ur + 32);
        tmem_ld_wait();
        reg_fence<64>(gr);
        reg_fence<64>(ur);
        if (c == 1) release();
        float *G = reinterpret_cast<float *>(gr);
        const float *U = reinterpret_cast<const float *>(ur);
#pragma unroll
        for (int i = 0; i < 64; ++i) G[i] = silu(G[i]) * U[i];
        sb[2 * c] = mx_block_words(G, cw + 16 * c);
        sb[2 * c + 1] = mx_block_words(G + 32, cw + 16 * c + 8);
      }
      if (store) {
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const int col = out_col + 64 * c;
          st.put(vQ, cw + 16 * c, col, row0, lane);
          *reinterpret_cast<uint16_t *>(g.outq_sf + sf_tiled_offset(grow, col / 32, g.ldq)) =
              static_cast<uint16_t>(sb[2 * c] | (sb[2 * c + 1] << 8));
        }
      }
      return;
    }
#pragma unroll 1
    for (int c = 0; c < 2; ++c) {
      uint32_t gr[64], ur[64];
      tmem_ld32_async(tb + 64 * c, gr);
      tmem_ld32_async(tb + 64 * c + 32, gr + 32);
      tmem_ld32_async(tb + 128 + 64 * c, ur);
      tmem_ld32_async(tb + 128 + 64 * c + 32, ur + 32);
      tmem_ld_wait();
      reg_fence<64>(gr);
      reg_fence<64>(ur);
      if (c == 1) release();
      if (!store) continue;
      float *G = reinterpret_cast<float *>(gr);
      float *U = reinterpret_cast<float *>(ur);
      const int col = out_col + 64 * c;
      if (g.out2) {
        st.put_bf16(vO2, G, col, row0, lane);
        st.put_bf16(vO2, G + 32, col + 32, row0, lane);
        st.put_bf16(vO2, U, g.m_half + col, row0, lane);
        st.put_bf16(vO2, U + 32, g.m_half + col + 32, row0, lane);
      }
#pragma unroll
      for (int i = 0; i < 64; ++i) G[i] = silu(G[i]) * U[i];  // h, in place
      if (g.out) {
        st.put_bf16(vO, G, col, row0, lane);
        st.put_bf16(vO, G + 32, col + 32, row0, lane);
      }
      if (g.outq) put_mx64(st, vQ, g.outq_sf, g.ldq, G, col, row0, grow, lane);
    }
  } else {  // EPI_SWIGLU_BWD: accumulator = dh; G|U saved in bf16
    constexpr int NCH = BN / 64;
#pragma unroll 1
    for (int c = 0; c < NCH; ++c) {
      uint32_t hr[64];
      tmem_ld32_async(tb + 64 * c, hr);
      tmem_ld32_async(tb + 64 * c + 32, hr + 32);
      tmem_ld_wait();
      reg_fence<64>(hr);
      if (c == NCH - 1) release();
      if (!store) continue;
      const float *dh = reinterpret_cast<const float *>(hr);
      const int col = out_col + 64 * c;
      float dG[64], dU[64];
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        float G[32], U[32];
        load_bf16x32(g.aux, grow, g.ld_aux, col + 32 * hh, G);
        load_bf16x32(g.aux, grow, g.ld_aux, g.m_half + col + 32 * hh, U);
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float d = dh[32 * hh + i];
          const float sg = sigmoidf(G[i]);
          dG[32 * hh + i] = round_bf16(d * U[i] * sg * (1.0f + G[i] * (1.0f - sg)));
          dU[32 * hh + i] = round_bf16(d * G[i] * sg);
        }
      }
      st.put_bf16(vO, dG, col, row0, lane);
      st.put_bf16(vO, dG + 32, col + 32, row0, lane);
      st.put_bf16(vO, dU, g.m_half + col, row0, lane);
      st.put_bf16(vO, dU + 32, g.m_half + col + 32, row0, lane);
      if (g.outq) {
        put_mx64(st, vQ, g.outq_sf, g.ldq, dG, col, row0, grow, lane);
        put_mx64(st, vQ, g.outq_sf, g.ldq, dU, g.m_half + col, row0, grow, lane);
      }
    }
  }
}

// SwiGLU backward of 32 dh columns of this lane's row (from column col of
// the tile's output): dG, dU from the saved bf16 G|U (read through aux),
// rounded to bf16; stores the bf16 values (g.out) and the column-blocked codes
// of dGU^T (g.outT), and returns the row-blocked MX codes of this block in
// cg[0..8) / cu[0..8) with their scale bytes.
MOE_DEV void swiglu_bwd32(const GemmArgs &g, const OutView &vO, Stager &st, const float *dh, int col, int row0,
                          long grow, int lane, uint32_t *cg, uint32_t *cu, uint32_t &sg, uint32_t &su) {
  float G[32], U[32];
  load_bf16x32(g.aux, grow, g.ld_aux, col, G);
  load_bf16x32(g.aux, grow, g.ld_aux, g.m_half + col, U);
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    const float d = dh[i];
    const float sgm = sigmoidf(G[i]);
    const float dg = round_bf16(d * U[i] * sgm * (1.0f + G[i] * (1.0f - sgm)));
    const float du = round_bf16(d * G[i] * sgm);
    G[i] = dg;
    U[i] = du;
  }
  if (g.out) {
    st.put_bf16(vO, G, col, row0, lane);
    st.put_bf16(vO, U, g.m_half + col, row0, lane);
  }
  // dG's codes first, then dU's, so that dG's values are dead while dU's
  // column codes are made (fewer registers live at once).
  if (g.outq) sg = mx_block_words(G, cg);
  if (g.outT)  // the gate/up wgrad operand dGU^T, column-blocked, from the bf16 dG, dU
    st.put_col_codes(G, g.outT, g.outT_sf, g.ldT, col, row0, lane);
  if (g.outq) su = mx_block_words(U, cu);
  if (g.outT) st.put_col_codes(U, g.outT, g.outT_sf, g.ldT, g.m_half + col, row0, lane);
}

// The row-blocked MX codes of 64 dG and 64 dU columns (two blocks each), with
// their scale bytes, for the gate/up dgrad.
MOE_DEV void swiglu_bwd_row_codes(const GemmArgs &g, const OutView &vQ, Stager &st, const uint32_t *cg,
                                  const uint32_t *cu, const uint32_t *sg, const uint32_t *su, int col, int row0,
                                  long grow, int lane) {
  if (!g.outq) return;
  st.put(vQ, cg, col, row0, lane);
  st.put(vQ, cu, g.m_half + col, row0, lane);
  *reinterpret_cast<uint16_t *>(g.outq_sf + sf_tiled_offset(grow, col / 32, g.ldq)) =
      static_cast<uint16_t>(sg[0] | (sg[1] << 8));
  *reinterpret_cast<uint16_t *>(g.outq_sf + sf_tiled_offset(grow, (g.m_half + col) / 32, g.ldq)) =
      static_cast<uint16_t>(su[0] | (su[1] << 8));
}

// Epilogue shared by two warps per TMEM lane quarter: warp `part` (0 or 1)
// drains half of the tile's columns.  For the store and SwiGLU epilogues the
// accumulator is read in one round (two warps in parallel) and released before
// any conversion or store; the SwiGLU backward reads its columns 64 at a time.
// STASH (one accumulator; SwiGLU backward): each warp keeps its first 32
// columns in registers, parks the rest in spare TMEM columns at ts, releases
// the accumulator, and reads the parked columns back 32 at a time, so fewer
// values are live at once (the 10-warp CTA has 168 registers per thread).
// DUMP (SwiGLU, a separate instantiation so the normal kernel carries none of
// its register pressure): also store the fp32 h to g.dump.
// NV (NVFP4 operands): the accumulator is multiplied by `sc` (the inverse of
// the operands' second-level scales) first, and the SwiGLU epilogue writes h
// as NVFP4 (store and SwiGLU epilogues only).
template <int EPI, int BN, bool DUMP = false, bool NV = false, bool STASH = false, typename Release>
MOE_DEV void epilogue_tile_split(const GemmArgs &g, const OutView &vO, const OutView &vO2,
                                 const OutView &vQ, Stager &st, uint32_t tb, int nk, int row0,
                                 long grow, int out_col, int lane, int part, bool store,
                                 Release release, float sc = 1.0f, uint32_t ts = 0) {
  if constexpr (EPI == EPI_STORE) {
    constexpr int NC = BN / 2;  // accumulator columns of this warp
    constexpr int NC32 = NC / 32;
    const int c0 = part * NC;
    if (nk == 0) {
      release();
      if (store) {
        float z[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) z[i] = 0.f;
#pragma unroll 1
        for (int c = 0; c < NC32; ++c) st.put_bf16(vO, z, out_col + c0 + 32 * c, row0, lane);
      }
      return;
    }
    // All of this warp's columns are read with back-to-back TMEM loads and one
    // wait, TMEM is released, and only then are they packed (in place) and
    // stored: the next tile's MMAs wait only for the loads.
    uint32_t raw[NC];
#pragma unroll
    for (int c = 0; c < NC32; ++c) tmem_ld32_async(tb + c0 + 32 * c, raw + 32 * c);
    tmem_ld_wait();
    reg_fence<NC>(raw);
    release();
    if constexpr (NV) {
#pragma unroll
      for (int i = 0; i < NC / 2; ++i)
        raw[i] = pack_bf16x2(__uint_as_float(raw[2 * i]) * sc, __uint_as_float(raw[2 * i + 1]) * sc);
    } else {
#pragma unroll
      for (int i = 0; i < NC / 2; ++i)
        raw[i] = pack_bf16x2(__uint_as_float(raw[2 * i]), __uint_as_float(raw[2 * i + 1]));
    }
    if (store) {
#pragma unroll
      for (int c = 0; c < NC32; ++c) st.put(vO, raw + 16 * c, out_col + c0 + 32 * c, row0, lane);
    }
  } else if constexpr (EPI == EPI_STORE_F32 || EPI == EPI_ADD_BF16) {
    // This warp's BN/2 columns in one round of TMEM loads, then TMEM is
    // released.  STORE_F32 writes the fp32 accumulator (16 values per 64-byte
    // piece); ADD_BF16 adds the current bf16 output row (read through aux, the
    // same buffer) and rounds the sum to bf16 once.
    constexpr int NC = BN / 2;
    const int c0 = part * NC;
    uint32_t raw[NC];
#pragma unroll
    for (int c = 0; c < NC / 32; ++c) tmem_ld32_async(tb + c0 + 32 * c, raw + 32 * c);
    tmem_ld_wait();
    reg_fence<NC>(raw);
    release();
    if (!store) return;
    if constexpr (EPI == EPI_STORE_F32) {
#pragma unroll
      for (int c = 0; c < NC / 16; ++c) st.put(vO, raw + 16 * c, out_col + c0 + 16 * c, row0, lane);
    } else {
      const bool in = grow < g.out_rows;
#pragma unroll
      for (int c = 0; c < NC / 32; ++c) {
        float v[32];
        if (in) {
          load_bf16x32(g.aux, grow, g.ld_aux, out_col + c0 + 32 * c, v);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = 0.f;
        }
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] += __uint_as_float(raw[32 * c + i]);
        st.put_bf16(vO, v, out_col + c0 + 32 * c, row0, lane);
      }
    }
  } else if constexpr (EPI == EPI_SWIGLU_BWD) {
    // This warp's BN/2 dh columns, 64 at a time (two 32-column halves).
    // Without STASH, each chunk is read from TMEM, then processed, and TMEM is
    // released once the last chunk has been read.  With STASH (one
    // accumulator), every 32-column piece but the first is copied into spare
    // TMEM columns at ts (this warp's lane quarter; BN/2 - 32 columns per
    // column half) and the accumulator is released, so the next tile's MMAs
    // overlap the processing; each piece is then read back when it is used,
    // which keeps 32 dh values in registers instead of 64.
    constexpr int NCH = BN / 128;
    if constexpr (STASH) {
      constexpr int NP = BN / 64;  // 32-column pieces of this warp
      const uint32_t a0 = tb + static_cast<uint32_t>(part * (BN / 2));
      const uint32_t stash = ts + static_cast<uint32_t>(part * 32 * (NP - 1));
      uint32_t h0[32];
      tmem_ld32_async(a0, h0);
#pragma unroll 1
      for (int p = 1; p < NP; ++p) {
        uint32_t t[32];
        tmem_ld32_async(a0 + 32 * p, t);
        tmem_ld_wait();
        reg_fence<32>(t);
        tmem_st32(stash + 32 * (p - 1), t);
      }
      tmem_ld_wait();
      reg_fence<32>(h0);
      tmem_st_wait();
      release();
      if (!store) return;
#pragma unroll
      for (int ch = 0; ch < NCH; ++ch) {
        const int col = out_col + part * (BN / 2) + 64 * ch;
        uint32_t cg[16], cu[16];  // MX codes of dG and dU (two blocks each)
        uint32_t sg[2], su[2];
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          uint32_t hr[32];
          if (ch == 0 && hh == 0) {
#pragma unroll
            for (int i = 0; i < 32; ++i) hr[i] = h0[i];
          } else {
            tmem_ld32_async(stash + 32 * (2 * ch + hh - 1), hr);
            tmem_ld_wait();
            reg_fence<32>(hr);
          }
          swiglu_bwd32(g, vO, st, reinterpret_cast<const float *>(hr), col + 32 * hh, row0, grow, lane,
                       cg + 8 * hh, cu + 8 * hh, sg[hh], su[hh]);
        }
        swiglu_bwd_row_codes(g, vQ, st, cg, cu, sg, su, col, row0, grow, lane);
      }
    } else {
#pragma unroll 1
      for (int ch = 0; ch < NCH; ++ch) {
        const int dc = part * (BN / 2) + 64 * ch;  // accumulator column of this chunk
        uint32_t hr[64];
        tmem_ld32_async(tb + dc, hr);
        tmem_ld32_async(tb + dc + 32, hr + 32);
        tmem_ld_wait();
        reg_fence<64>(hr);
        if (ch == NCH - 1) release();
        if (!store) continue;
        const int col = out_col + dc;
        uint32_t cg[16], cu[16];
        uint32_t sg[2], su[2];
#pragma unroll
        for (int hh = 0; hh < 2; ++hh)
          swiglu_bwd32(g, vO, st, reinterpret_cast<const float *>(hr) + 32 * hh, col + 32 * hh, row0, grow, lane,
                       cg + 8 * hh, cu + 8 * hh, sg[hh], su[hh]);
        swiglu_bwd_row_codes(g, vQ, st, cg, cu, sg, su, col, row0, grow, lane);
      }
    }
  } else {  // EPI_SWIGLU: accumulator [0,128) = G, [128,256) = U; this warp: 64 h columns
    const int hc = part * 64;
    uint32_t gr[64], ur[64];
    tmem_ld32_async(tb + hc, gr);
    tmem_ld32_async(tb + hc + 32, gr + 32);
    tmem_ld32_async(tb + 128 + hc, ur);
    tmem_ld32_async(tb + 128 + hc + 32, ur + 32);
    tmem_ld_wait();
    reg_fence<64>(gr);
    reg_fence<64>(ur);
    release();
    if (!store) return;
    float *G = reinterpret_cast<float *>(gr);
    float *U = reinterpret_cast<float *>(ur);
    if constexpr (NV) {
#pragma unroll
      for (int i = 0; i < 64; ++i) {
        G[i] *= sc;
        U[i] *= sc;
      }
    }
    const int col = out_col + hc;
    if (g.out2) {
      st.put_bf16(vO2, G, col, row0, lane);
      st.put_bf16(vO2, G + 32, col + 32, row0, lane);
      st.put_bf16(vO2, U, g.m_half + col, row0, lane);
      st.put_bf16(vO2, U + 32, g.m_half + col + 32, row0, lane);
    }
#pragma unroll
    for (int i = 0; i < 64; ++i) G[i] = silu(G[i]) * U[i];  // h, in place
    if constexpr (DUMP) {  // test hook: the fp32 h the quantisers below read
      if (grow < g.out_rows) {
        float4 *dst = reinterpret_cast<float4 *>(g.dump + grow * g.ld_dump + col);
#pragma unroll
        for (int i = 0; i < 16; ++i) dst[i] = make_float4(G[4 * i], G[4 * i + 1], G[4 * i + 2], G[4 * i + 3]);
      }
    }
    if (g.out) {
      st.put_bf16(vO, G, col, row0, lane);
      st.put_bf16(vO, G + 32, col + 32, row0, lane);
    }
    if (g.outT) {  // the wgrad operand h^T, column-blocked, from the bf16 h
      st.put_col_codes(G, g.outT, g.outT_sf, g.ldT, col, row0, lane);
      st.put_col_codes(G + 32, g.outT, g.outT_sf, g.ldT, col + 32, row0, lane);
    }
    if (g.outq) {
      if constexpr (NV) put_nv64(g, G, col, grow);
      else put_mx64(st, vQ, g.outq_sf, g.ldq, G, col, row0, grow, lane);
    }
  }
}

}  // namespace gemm_detail
}  // namespace moe
