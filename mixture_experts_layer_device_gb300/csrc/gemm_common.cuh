// Epilogue helpers shared by the 1-CTA and 2-CTA grouped GEMM kernels.
#pragma once

#include "common.cuh"
#include "kernels.h"

namespace moe {
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

// Per-warp writer of 32-row x 64-byte output pieces: each lane places its row's
// 64 bytes in a 64-byte-swizzled shared-memory buffer (conflict-free), then one
// lane stores the box with TMA.  With several buffers the staging of one piece
// overlaps the stores of the previous ones; a buffer is reused only after the
// store that last read it has finished reading shared memory.
struct Stager {
  uint8_t *buf;  // nbuf x 2 KB, 512-byte aligned
  int n;
  int nbuf;      // 1, 2 or 4
  MOE_DEV Stager(uint8_t *b, int buffers) : buf(b), n(0), nbuf(buffers) {}
  MOE_DEV void put(const CUtensorMap *map, const uint32_t *w16, int c0, int row0, int lane) {
    uint8_t *half = buf + (n & (nbuf - 1)) * 2048;
    if (lane == 0 && n >= nbuf) {
      if (nbuf == 4) bulk_wait_read<3>();
      else if (nbuf == 2) bulk_wait_read<1>();
      else bulk_wait_read<0>();
    }
    __syncwarp();
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int jj = j ^ ((lane >> 1) & 3);
      *reinterpret_cast<uint4 *>(half + lane * 64 + jj * 16) =
          make_uint4(w16[4 * j], w16[4 * j + 1], w16[4 * j + 2], w16[4 * j + 3]);
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      tma_store_2d(map, half, c0, row0);
      bulk_commit();
    }
    ++n;
  }
  MOE_DEV void put_bf16(const CUtensorMap *map, const float *v32, int c0, int row0, int lane) {
    uint32_t w[16];
    bf16x32_words(v32, w);
    put(map, w, c0, row0, lane);
  }
};

// Two MX blocks (64 values) of one row -> one 64-byte codes piece + 2 scale bytes.
MOE_DEV void put_mx64(Stager &st, const CUtensorMap *map, uint8_t *sf, long ldq, const float *v64,
                      int col, int row0, long grow, int lane) {
  uint32_t w[16];
  const uint32_t b0 = mx_block_words(v64, w);
  const uint32_t b1 = mx_block_words(v64 + 32, w + 8);
  st.put(map, w, col, row0, lane);
  // (col / 32) is even, so both bytes sit next to each other in one 512-byte atom.
  *reinterpret_cast<uint16_t *>(sf + sf_tiled_offset(grow, col / 32, ldq)) =
      static_cast<uint16_t>(b0 | (b1 << 8));
}


// Drains one tile's accumulator (this warp's 32 TMEM lanes at `tb`) and writes
// the epilogue's outputs with TMA stores.  `release()` is called once the last
// accumulator column has been read (the MMA may then reuse it).  With
// store == false the accumulator is drained and released but nothing is
// written (the idle half of a 2-CTA tile).
template <int EPI, int BN, typename Release>
MOE_DEV void epilogue_tile(const GemmArgs &g, const CUtensorMap *tmO, const CUtensorMap *tmO2,
                           const CUtensorMap *tmQ, Stager &st, uint32_t tb, int nk, int row0,
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
        for (int c = 0; c < 2 * NCH; ++c) st.put_bf16(tmO, z, out_col + 32 * c, row0, lane);
      }
      return;
    }
    // The whole row is drained into registers as packed bf16 pairs (TMEM loads
    // of 32 columns ping-pong with the conversion), TMEM is released, and only
    // then are the pieces staged and stored: the accumulator is never held
    // while TMA stores queue behind the producer's loads.
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
      for (int c = 0; c < NC32; ++c) st.put(tmO, pk + 16 * c, out_col + 32 * c, row0, lane);
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
          st.put(tmQ, cw + 16 * c, col, row0, lane);
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
        st.put_bf16(tmO2, G, col, row0, lane);
        st.put_bf16(tmO2, G + 32, col + 32, row0, lane);
        st.put_bf16(tmO2, U, g.m_half + col, row0, lane);
        st.put_bf16(tmO2, U + 32, g.m_half + col + 32, row0, lane);
      }
#pragma unroll
      for (int i = 0; i < 64; ++i) G[i] = silu(G[i]) * U[i];  // h, in place
      if (g.out) {
        st.put_bf16(tmO, G, col, row0, lane);
        st.put_bf16(tmO, G + 32, col + 32, row0, lane);
      }
      if (g.outq) put_mx64(st, tmQ, g.outq_sf, g.ldq, G, col, row0, grow, lane);
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
      st.put_bf16(tmO, dG, col, row0, lane);
      st.put_bf16(tmO, dG + 32, col + 32, row0, lane);
      st.put_bf16(tmO, dU, g.m_half + col, row0, lane);
      st.put_bf16(tmO, dU + 32, g.m_half + col + 32, row0, lane);
      if (g.outq) {
        put_mx64(st, tmQ, g.outq_sf, g.ldq, dG, col, row0, grow, lane);
        put_mx64(st, tmQ, g.outq_sf, g.ldq, dU, g.m_half + col, row0, grow, lane);
      }
    }
  }
}

// Epilogue shared by two warps per TMEM lane quarter: warp `part` (0 or 1)
// drains half of the tile's columns.  The accumulator is read in one round
// (two warps in parallel) and released before any conversion or store.
// EPI_SWIGLU_BWD needs BN = 128 here (64 dh columns per warp).
template <int EPI, int BN, typename Release>
MOE_DEV void epilogue_tile_split(const GemmArgs &g, const CUtensorMap *tmO, const CUtensorMap *tmO2,
                                 const CUtensorMap *tmQ, Stager &st, uint32_t tb, int nk, int row0,
                                 long grow, int out_col, int lane, int part, bool store,
                                 Release release) {
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
        for (int c = 0; c < NC32; ++c) st.put_bf16(tmO, z, out_col + c0 + 32 * c, row0, lane);
      }
      return;
    }
    uint32_t pk[NC / 2];
    uint32_t buf[2][32];
    tmem_ld32_async(tb + c0, buf[0]);
    tmem_ld_wait();
    reg_fence<32>(buf[0]);
#pragma unroll
    for (int c = 0; c < NC32; ++c) {
      if (c + 1 < NC32) tmem_ld32_async(tb + c0 + 32 * (c + 1), buf[(c + 1) & 1]);
      bf16x32_words(reinterpret_cast<const float *>(buf[c & 1]), pk + 16 * c);
      if (c + 1 < NC32) {
        tmem_ld_wait();
        reg_fence<32>(buf[(c + 1) & 1]);
      }
    }
    release();
    if (store) {
#pragma unroll
      for (int c = 0; c < NC32; ++c) st.put(tmO, pk + 16 * c, out_col + c0 + 32 * c, row0, lane);
    }
  } else if constexpr (EPI == EPI_SWIGLU_BWD) {
    static_assert(BN == 128, "split SwiGLU-backward epilogue expects 128-column tiles");
    const int dc = part * 64;  // this warp's 64 dh columns
    uint32_t hr[64];
    tmem_ld32_async(tb + dc, hr);
    tmem_ld32_async(tb + dc + 32, hr + 32);
    tmem_ld_wait();
    reg_fence<64>(hr);
    release();
    if (!store) return;
    const float *dh = reinterpret_cast<const float *>(hr);
    const int col = out_col + dc;
    uint32_t cg[16], cu[16];  // MX codes of dG and dU (two blocks each)
    uint32_t sg[2], su[2];
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      float G[32], U[32];
      load_bf16x32(g.aux, grow, g.ld_aux, col + 32 * hh, G);
      load_bf16x32(g.aux, grow, g.ld_aux, g.m_half + col + 32 * hh, U);
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const float d = dh[32 * hh + i];
        const float sgm = sigmoidf(G[i]);
        const float dg = round_bf16(d * U[i] * sgm * (1.0f + G[i] * (1.0f - sgm)));
        const float du = round_bf16(d * G[i] * sgm);
        G[i] = dg;
        U[i] = du;
      }
      st.put_bf16(tmO, G, col + 32 * hh, row0, lane);
      st.put_bf16(tmO, U, g.m_half + col + 32 * hh, row0, lane);
      if (g.outq) {
        sg[hh] = mx_block_words(G, cg + 8 * hh);
        su[hh] = mx_block_words(U, cu + 8 * hh);
      }
    }
    if (g.outq) {
      st.put(tmQ, cg, col, row0, lane);
      st.put(tmQ, cu, g.m_half + col, row0, lane);
      *reinterpret_cast<uint16_t *>(g.outq_sf + sf_tiled_offset(grow, col / 32, g.ldq)) =
          static_cast<uint16_t>(sg[0] | (sg[1] << 8));
      *reinterpret_cast<uint16_t *>(g.outq_sf + sf_tiled_offset(grow, (g.m_half + col) / 32, g.ldq)) =
          static_cast<uint16_t>(su[0] | (su[1] << 8));
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
    const float *U = reinterpret_cast<const float *>(ur);
    const int col = out_col + hc;
    if (g.out2) {
      st.put_bf16(tmO2, G, col, row0, lane);
      st.put_bf16(tmO2, G + 32, col + 32, row0, lane);
      st.put_bf16(tmO2, U, g.m_half + col, row0, lane);
      st.put_bf16(tmO2, U + 32, g.m_half + col + 32, row0, lane);
    }
#pragma unroll
    for (int i = 0; i < 64; ++i) G[i] = silu(G[i]) * U[i];  // h, in place
    if (g.out) {
      st.put_bf16(tmO, G, col, row0, lane);
      st.put_bf16(tmO, G + 32, col + 32, row0, lane);
    }
    if (g.outq) put_mx64(st, tmQ, g.outq_sf, g.ldq, G, col, row0, grow, lane);
  }
}

}  // namespace gemm_detail
}  // namespace moe
