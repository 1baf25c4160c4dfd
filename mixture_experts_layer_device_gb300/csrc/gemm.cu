// Grouped expert GEMMs on the 5th-generation tensor cores (tcgen05 + TMEM).
//
// D[128 x BN] = A[128 x K] * B[BN x K]^T per tile, both operands K-major,
// moved by TMA into 128-byte-swizzled shared memory, multiplied by one thread
// issuing tcgen05.mma into a TMEM accumulator, and drained by four epilogue
// warps with tcgen05.ld.  BF16 (kind::f16) or OCP MXFP8 (kind::mxf8f6f4 with
// E8M0 block scales copied into TMEM by tcgen05.cp).
//
// Method references ("Mixture-of-Kittens" wiki page): expert grouped GEMMs in
// MXFP8 with SwiGLU and quantisation fused (flowchart, Key claims MXFP8
// bullet); a persistent kernel whose roles hand off through counters rather
// than a global barrier (TL;DR) -- here the roles are warps of one CTA and the
// counters are shared-memory mbarriers.
//
// Tile schedules:
//   GROUP_M  rows of A are expert-sorted and padded per expert to 128, so every
//            128-row tile belongs to one expert; B is that expert's weights.
//            Tiles of one expert are consecutive (m-tile major), which keeps
//            the expert's weight panel hot in L2 while its rows stream.
//            When the load is bimodal -- a few experts with many m-tiles and
//            the rest with one or two -- the light experts' tiles (which
//            stream their weight panel from HBM for at most 256 rows) are
//            spread evenly among the heavy experts' tiles (which re-read
//            theirs from L2), each kind still in expert order, so HBM streams
//            while the tensor cores work; their B loads carry L2 evict-first
//            and the heavy experts' evict-last, so the streamed panels do not
//            push the heavy panels out of L2.
//   DENSE    one group (shared expert).
//   GROUP_K  weight gradients: the reduction runs over one expert's padded
//            rows [poff[e], poff[e+1]) of two transposed operands.  An
//            expert with no rows gets all-zero tiles, or, with skip_empty,
//            no tiles at all (a plain store kernel writes its zeros).
// Every output element is produced by one CTA with a fixed K order, so results
// are bitwise reproducible.
#include "common.cuh"
#include "dispatch_tile.cuh"
#include "gemm_common.cuh"
#include "kernels.h"

namespace moe {

namespace {

using namespace gemm_detail;

// Operand formats of the single-CTA GEMM: BF16 (kind::f16), MXFP8 (E4M3 with
// an E8M0 scale per 32 along K, kind::mxf8f6f4) and NVFP4 (packed E2M1 with an
// E4M3 scale per 16 along K, kind::mxf4nvf4 with scale_vec::4X; the
// accumulator is multiplied by the two operands' second-level scales in the
// epilogue).  Every format moves 128-byte rows of A and B per stage.
template <int F, int BN>
struct Cfg {
  static constexpr bool MX = F != FMT_BF16;  // block-scaled operands
  static constexpr bool NV = F == FMT_NVFP4;
  static constexpr int BM = 128;
  static constexpr int BK = NV ? 256 : (MX ? 128 : 64);  // elements per 128-byte smem row
  static constexpr int UK = NV ? 64 : (MX ? 32 : 16);    // K per tcgen05.mma
  static constexpr int KSTEPS = BK / UK;
  static constexpr int A_BYTES = BM * 128;
  static constexpr int B_BYTES = BN * 128;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  // 512-byte scale atoms (128 rows x 4 blocks) per 128 rows and stage: one
  // MXFP8 atom spans 128 of K, an NVFP4 atom 64, so an NVFP4 stage needs four
  static constexpr int SF_ATOMS = NV ? 4 : 1;
  static constexpr int STAGES = NV ? (BN == 256 ? 3 : 5) : (BN == 256 ? 4 : 6);
  static constexpr int SFA_BYTES = MX ? 512 * SF_ATOMS : 0;
  static constexpr int SFB_BYTES = MX ? (BN / 128) * 512 * SF_ATOMS : 0;
  static constexpr int SF_STAGE = SFA_BYTES + SFB_BYTES;
  static constexpr int NUM_ACC = (MX && BN == 256) ? 1 : 2;
  static constexpr uint32_t TMEM_COLS = 512;
  // Scale factors get their own TMEM columns per pipeline stage (4 for A, BN/32
  // for B, per atom), so copying a stage's scales never waits for the MMAs
  // still reading the previous stage's.  MMA k of an NVFP4 stage reads atom k:
  // A at columns 4k, B at 4 SF_ATOMS + k BN/32 of the stage's block.
  static constexpr int SFA_COLS = 4 * SF_ATOMS;
  static constexpr int SF_COLS = SF_ATOMS * (4 + BN / 32);
  static constexpr int SF_COL0 = NUM_ACC * BN;
  // The SwiGLU-backward epilogue's stash (one accumulator only): every
  // 32-column piece of the accumulator but each warp's first, the last
  // 2 x 32 (BN / 64 - 1) columns of TMEM.
  static constexpr bool STASH = !NV && NUM_ACC == 1 && BN / 128 > 1;  // NVFP4 has no backward
  static constexpr int STASH_COL = 512 - 2 * 32 * (BN / 64 - 1);
  static constexpr uint32_t TX_BYTES = STAGE_BYTES + SF_STAGE;
  static constexpr uint32_t IDESC = NV ? idesc_nvf4(128, BN) : (MX ? idesc_mxf8(128, BN) : idesc_bf16(128, BN));
  // epilogue staging: 2 KB pieces (32 rows x 64 B, 64-byte swizzle), 16 KB split
  // over the epilogue warps
  static constexpr int STAGING_BYTES = 4 * 4096;
  // barriers: full[S], empty[S], tfull[NA], tempty[NA], done
  static constexpr int NBAR = 2 * STAGES + 2 * NUM_ACC + 1;
  static constexpr size_t SMEM = 1024 + static_cast<size_t>(STAGES) * (STAGE_BYTES + SF_STAGE) +
                                 STAGING_BYTES + NBAR * 8 + 16;
  static_assert(!MX || SF_COL0 + STAGES * SF_COLS <= 512, "TMEM columns");
  static_assert(!STASH || SF_COL0 + (MX ? STAGES * SF_COLS : 0) <= STASH_COL, "TMEM columns of the stash");
  static_assert(NUM_ACC * BN <= 512, "TMEM columns");
  // dynamic + the kernel's static shared memory (the interleave tables)
  static_assert(SMEM + 8 * 1025 + 16 <= 232448, "shared memory");
};

struct Tile {
  int a_row, k0, nk, b_row0, b_row1, out_row, out_col;
  int e;  // group (expert) of the tile
  bool light;  // GROUP_M, interleaved order: a light expert's tile
};

// Interleaved GROUP_M order: experts with fewer than kLightMTiles m-tiles are
// light; it is used when every other active expert has at least
// kHeavyMinMTiles m-tiles (a bimodal load) and E <= kMaxInterleaveE.
constexpr int kLightMTiles = 3;
constexpr int kHeavyMinMTiles = 16;
constexpr int kMaxInterleaveE = 1024;

template <int BK, int BN, int EPI>
MOE_DEV int total_tiles(const GemmArgs &g) {
  if (g.sched == SCHED_GROUP_M) return g.n_tiles * (__ldg(g.poff + g.E) >> 7);
  if (g.sched == SCHED_DENSE) return g.n_tiles * ((g.M + 127) >> 7);
  return g.E * (g.M >> 7) * g.n_tiles;
}

// il (GROUP_M, interleaved order, else NULL): the exclusive prefix sums of the
// heavy experts' m-tiles [E + 1] followed by the light experts' [E + 1].  Tile
// t is light when floor((t + 1) L / T) > floor(t L / T) (T tiles, L of them
// light), so the light tiles are spread evenly; the number before t indexes the
// light order, the rest the heavy order.
template <int BK, int BN, int EPI>
MOE_DEV Tile decode_tile(const GemmArgs &g, int t, const int *il) {
  Tile ti;
  ti.light = false;
  const int nt = g.n_tiles;
  int e = 0, mt, ntile;
  if (g.sched == SCHED_GROUP_M && il) {
    const int *hoff = il, *loff = il + g.E + 1;
    const long LT = static_cast<long>(loff[g.E]) * nt;
    const long TT = static_cast<long>(hoff[g.E] + loff[g.E]) * nt;
    const long j0 = static_cast<long>(t) * LT / TT;
    const long j1 = static_cast<long>(t + 1) * LT / TT;
    ti.light = j1 > j0;
    const int idx = ti.light ? static_cast<int>(j0) : t - static_cast<int>(j0);
    const int *off = ti.light ? loff : hoff;
    const int lm = idx / nt;
    ntile = idx % nt;
    int lo = 0, hi = g.E - 1;  // the last expert whose range starts at or before lm
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (off[mid] <= lm) lo = mid;
      else hi = mid - 1;
    }
    e = lo;
    mt = lm - off[e];
    ti.a_row = ((__ldg(g.poff + e) >> 7) + mt) * 128;
    ti.k0 = 0;
    ti.nk = g.K / BK;
    ti.out_row = ti.a_row;
  } else if (g.sched == SCHED_GROUP_M) {
    int lo = 0, hi = g.E - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (nt * (__ldg(g.poff + mid) >> 7) <= t) lo = mid;
      else hi = mid - 1;
    }
    e = lo;
    const int ms = __ldg(g.poff + e) >> 7;
    const int local = t - nt * ms;
    mt = local / nt;
    ntile = local % nt;
    ti.a_row = (ms + mt) * 128;
    ti.k0 = 0;
    ti.nk = g.K / BK;
    ti.out_row = ti.a_row;
  } else if (g.sched == SCHED_DENSE) {
    mt = t / nt;
    ntile = t % nt;
    ti.a_row = mt * 128;
    ti.k0 = 0;
    ti.nk = g.K / BK;
    ti.out_row = ti.a_row;
  } else {
    const int mtn = (g.M >> 7) * nt;
    e = t / mtn;
    const int r = t % mtn;
    mt = r / nt;
    ntile = r % nt;
    ti.a_row = mt * 128;
    if (g.poff) {
      ti.k0 = __ldg(g.poff + e);
      ti.nk = (__ldg(g.poff + e + 1) - ti.k0) / BK;
    } else {
      ti.k0 = 0;
      ti.nk = g.K / BK;
    }
    ti.out_row = e * g.M + mt * 128;
  }
  ti.e = e;
  if (EPI == EPI_SWIGLU) {
    ti.b_row0 = e * g.b_rows_per_group + ntile * 128;
    ti.b_row1 = ti.b_row0 + g.b_split;
    ti.out_col = ntile * 128;
  } else {
    ti.b_row0 = (g.sched == SCHED_GROUP_K ? 0 : e * g.b_rows_per_group) + ntile * BN;
    ti.b_row1 = ti.b_row0 + 128;
    ti.out_col = ntile * BN;
  }
  return ti;
}

// Gather role of the ring kernel: data movement only.  The row-blocked codes
// of every token were computed once beforehand (xq, with canonical scales
// xq_sf); a gather CTA copies the rows of tiles u = blockIdx.x, + gather_ctas,
// ... (increasing) into their ring slots:
//   warp 8: whole rows, 4 at a time (lane i < 4 moves row i of the group),
//     with TMA bulk copies global -> shared and shared -> ring (a zero row
//     for padding rows); 6 buffers, the loads of the next 4 groups in flight
//     while one is stored.  Whole-row copies keep the number of TMA
//     operations per tile at 2 x 128;
//   warps 0..7: scatter each row's scale bytes into the slot's tiled layout
//     (16 loads in flight per thread before the stores).
// Before the first write of tile u into slot u % slots the slot's previous
// tile (u - slots) must have been loaded by all n_tiles GEMM tiles that read
// it; once the tile's copies are complete the slot is published with
// ready[slot] = u + 1 (release).  The codes are those of the stand-alone
// dispatch (row-blocked quantisation along d depends only on the token).
namespace ring {
constexpr int NBUF = 6;
constexpr int LAG = 4;          // groups loaded ahead of the one being stored
constexpr int GROUP = 4;        // rows per buffer
constexpr int MAX_D = 8192;     // codes per row (the ring needs d <= MAX_D)
constexpr int BUF_BYTES = GROUP * MAX_D;
constexpr int SF_BATCH = 16;
static_assert(NBUF - LAG - 1 == 1, "the buffer-reuse wait below assumes one newer store");
}  // namespace ring

MOE_DEV void ring_gather_role(const GemmArgs &g, uint8_t *smem) {
  using namespace ring;
  const RingArgs &r = g.ring;
  const int tid = static_cast<int>(threadIdx.x);
  const int warp = tid >> 5, lane = tid & 31;
  const int d = g.K;
  uint8_t *bufs = smem;                                     // NBUF x GROUP rows of d bytes
  uint8_t *zrow = smem + NBUF * GROUP * d;                  // d zero bytes
  int *toks = reinterpret_cast<int *>(zrow + d);            // 128 tokens of the current tile
  uint64_t *full = reinterpret_cast<uint64_t *>(toks + 128);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(full + NBUF);
  volatile int *stop = abort_flag + 1;
  for (int i = tid; i < d / 16; i += blockDim.x) reinterpret_cast<uint4 *>(zrow)[i] = make_uint4(0, 0, 0, 0);
  if (tid == 0) {
    for (int b = 0; b < NBUF; ++b) mbar_init(&full[b], 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  fence_proxy_async_smem();  // the zero row is read by TMA stores
  __syncthreads();
  if (g.debug_starve) return;  // test hook: nothing is published, the GEMM CTAs' ring waits run out

  constexpr int items = 128 / GROUP;  // row groups of one tile
  const int ngrp = d / 128;           // 4-byte scale groups per row
  const int tiles = __ldg(r.rb.poff + g.E) >> 7;
  int gi = 0;                         // buffer uses so far (warp 8)
  for (int u = static_cast<int>(blockIdx.x); u < tiles; u += r.gather_ctas) {
    const int slot = u % r.slots;
    if (tid < 128) toks[tid] = token_of_row(r.rb, g.E, r.k, u * 128 + tid, nullptr);
    if (tid == 0)
      *stop = flag_wait_geq(r.freed + slot, (u / r.slots) * g.n_tiles, r.abort, abort_flag, g.status,
                            g.timeout_ns)
                  ? 0
                  : 1;
    __syncthreads();
    if (*stop) break;
    uint8_t *dst_rows = r.codes + static_cast<size_t>(slot) * 128 * d;
    if (warp == 8) {
      // ---------------------------------------------- codes: TMA in, TMA out
      // Group j of this tile uses buffer (g0 + j) % NBUF; it is loaded in
      // iteration j and stored in iteration j + LAG.  The buffer's previous
      // group (j - NBUF) was stored in iteration j - NBUF + LAG = j - 2, so
      // before the load at most one newer store of this lane may still be
      // reading shared memory (NBUF - LAG - 1 = 1).
      const int g0 = gi;
      bool ok = true;
      for (int j = 0; j < items + LAG && ok; ++j) {
        if (j < items) {
          const int b = (g0 + j) % NBUF;
          const int tok = lane < GROUP ? toks[j * GROUP + lane] : -1;
          if (g0 + j >= NBUF) bulk_wait_read<NBUF - LAG - 1>();
          const unsigned valid = __ballot_sync(0xffffffffu, tok >= 0);
          if (lane == 0) mbar_arrive_expect_tx(&full[b], static_cast<uint32_t>(__popc(valid)) * d);
          __syncwarp();
          if (tok >= 0)
            bulk_load(bufs + (b * GROUP + lane) * d, r.xq + static_cast<size_t>(tok) * d,
                      static_cast<uint32_t>(d), &full[b]);
        }
        if (j >= LAG) {  // store group j - LAG
          const int jp = j - LAG;
          const int b = (g0 + jp) % NBUF;
          const uint32_t ph = static_cast<uint32_t>((g0 + jp) / NBUF) & 1u;
          ok = mbar_wait(&full[b], ph, abort_flag, g.status, g.timeout_ns);
          ok = __all_sync(0xffffffffu, ok);
          if (ok && lane < GROUP) {
            const int tok = toks[jp * GROUP + lane];
            bulk_store(dst_rows + static_cast<size_t>(jp * GROUP + lane) * d,
                       tok >= 0 ? bufs + (b * GROUP + lane) * d : zrow, static_cast<uint32_t>(d));
            bulk_commit();
          }
        }
      }
      gi = g0 + items;
      bulk_wait<0>();  // this lane's ring writes are complete
      fence_proxy_async_global();
      __threadfence();
      if (!ok) *abort_flag = 1;
    } else if (warp < 8) {
      // ---------------------------------------------- scales: canonical -> tiled
      const int rows_sf = slot * 128;
      const int total = 128 * ngrp;
      for (int base = 0; base < total; base += 256 * SF_BATCH) {
        uint32_t v[SF_BATCH];
#pragma unroll
        for (int q = 0; q < SF_BATCH; ++q) {
          const int i = base + q * 256 + tid;
          v[q] = 0u;
          if (i < total) {
            const int tok = toks[i / ngrp];
            if (tok >= 0)
              v[q] = __ldg(reinterpret_cast<const uint32_t *>(r.xq_sf + static_cast<size_t>(tok) * (d / 32) +
                                                               4 * (i % ngrp)));
          }
        }
#pragma unroll
        for (int q = 0; q < SF_BATCH; ++q) {
          const int i = base + q * 256 + tid;
          if (i < total)
            *reinterpret_cast<uint32_t *>(r.sf + sf_tiled_offset(rows_sf + i / ngrp, 4 * (i % ngrp), d)) = v[q];
        }
      }
      __threadfence();
      fence_proxy_async_global();
    }
    __syncthreads();
    if (*abort_flag) break;
    if (tid == 0) st_release_gpu(r.ready + slot, u + 1);
  }
}

// Epilogue warps per CTA: 8, two per TMEM lane quarter, each draining half of
// the columns (the SwiGLU backward 64 columns at a time, so its per-row working
// set fits the registers of 320 threads at any tile width).
template <int EPI, int BN>
__host__ __device__ constexpr int epi_warps() {
  return 8;
}

template <int F, int BN, int EPI, bool RING = false, bool DUMP = false>
__global__ void __launch_bounds__(64 + 32 * epi_warps<EPI, BN>(), 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const GemmArgs g) {
  using C = Cfg<F, BN>;
  constexpr bool MX = C::MX;
  constexpr bool NV = C::NV;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  if constexpr (RING) {
    if (static_cast<int>(blockIdx.x) < g.ring.gather_ctas) {
      ring_gather_role(g, smem);
      return;
    }
  }
  // GEMM CTAs: this one's index among them and their number
  const int cta = static_cast<int>(blockIdx.x) - (RING ? g.ring.gather_ctas : 0);
  const int ncta = static_cast<int>(gridDim.x) - (RING ? g.ring.gather_ctas : 0);
  uint8_t *sf_base = smem + C::STAGES * C::STAGE_BYTES;
  uint8_t *staging = sf_base + C::STAGES * C::SF_STAGE;
  uint64_t *bars = reinterpret_cast<uint64_t *>(staging + C::STAGING_BYTES);
  uint64_t *full = bars;
  uint64_t *empty = bars + C::STAGES;
  uint64_t *tfull = bars + 2 * C::STAGES;
  uint64_t *tempty = tfull + C::NUM_ACC;
  uint64_t *done = tempty + C::NUM_ACC;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(done + 1);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < C::NUM_ACC; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 32 * epi_warps<EPI, BN>());
    }
    mbar_init(done, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  // Interleaved GROUP_M order: prefix sums of the heavy and light experts'
  // m-tiles and the bimodality test, by one epilogue warp before the roles
  // split (the ring's tiles keep expert order).
  __shared__ int il_off[2 * (kMaxInterleaveE + 1)];
  __shared__ int il_on;
  if (warp == 2) {
    bool on = false;
    if (!RING && g.sched == SCHED_GROUP_M && g.E <= kMaxInterleaveE) {
      int runh = 0, runl = 0, min_heavy = 1 << 30;
      for (int base = 0; base < g.E; base += 32) {
        const int e = base + lane;
        const int c = e < g.E ? (__ldg(g.poff + e + 1) >> 7) - (__ldg(g.poff + e) >> 7) : 0;
        const int ch = c >= kLightMTiles ? c : 0;
        const int cl = c >= kLightMTiles ? 0 : c;
        int ih = ch, il_inc = cl, mn = ch > 0 ? ch : (1 << 30);
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int a = __shfl_up_sync(0xffffffffu, ih, o);
          const int b = __shfl_up_sync(0xffffffffu, il_inc, o);
          if (lane >= o) {
            ih += a;
            il_inc += b;
          }
          mn = min(mn, __shfl_xor_sync(0xffffffffu, mn, o));
        }
        if (e < g.E) {
          il_off[e] = runh + ih - ch;
          il_off[g.E + 1 + e] = runl + il_inc - cl;
        }
        runh += __shfl_sync(0xffffffffu, ih, 31);
        runl += __shfl_sync(0xffffffffu, il_inc, 31);
        min_heavy = min(min_heavy, mn);
      }
      if (lane == 0) {
        il_off[g.E] = runh;
        il_off[2 * g.E + 1] = runl;
      }
      on = runh > 0 && runl > 0 && min_heavy >= kHeavyMinMTiles;
    }
    if (lane == 0) il_on = on ? 1 : 0;
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int *il = il_on ? il_off : nullptr;
  const int total = total_tiles<C::BK, BN, EPI>(g);

  if (warp == 0) {
    // ------------------------------------------------ TMA producer
    if (lane == 0) {
      prefetch_tensormap(&tmA);
      prefetch_tensormap(&tmB);
      int stage = 0;
      uint32_t ph = 0;
      int armed[C::STAGES];
      for (int s = 0; s < C::STAGES; ++s) armed[s] = -1;
      for (int i = cta; i < total && !*abort_flag && (RING || !g.debug_starve); i += ncta) {
        const Tile ti = decode_tile<C::BK, BN, EPI>(g, i, il);
        int a_row = ti.a_row;  // row of A to load (the tile's ring slot with a ring)
        if constexpr (RING) {
          const int u = ti.a_row >> 7;
          const int slot = u % g.ring.slots;
          if (!flag_wait_geq(g.ring.ready + slot, u + 1, g.ring.abort, abort_flag, g.status, g.timeout_ns))
            break;
          fence_proxy_async_global();
          a_row = slot * 128;
        }
        for (int kb = 0; kb < ti.nk; ++kb) {
          if (!mbar_wait(&empty[stage], ph ^ 1u, abort_flag, g.status, g.timeout_ns)) break;
          uint8_t *sa = smem + stage * C::STAGE_BYTES;
          uint8_t *sb = sa + C::A_BYTES;
          mbar_arrive_expect_tx(&full[stage], C::TX_BYTES);
          armed[stage] = static_cast<int>(ph);
          const int kc = ti.k0 + kb * C::BK;
          const int kx = NV ? kc / 2 : kc;  // tensor-map coordinate: NVFP4 maps count bytes
          tma_load_2d(&tmA, &full[stage], sa, kx, a_row);
          if (il) {  // interleaved: streamed light panels leave L2 first
            const uint64_t pol = ti.light ? l2_policy_evict_first() : l2_policy_evict_last();
            tma_load_2d_hint(&tmB, &full[stage], sb, kx, ti.b_row0, pol);
            if (BN == 256) tma_load_2d_hint(&tmB, &full[stage], sb + 128 * 128, kx, ti.b_row1, pol);
          } else {
            tma_load_2d(&tmB, &full[stage], sb, kx, ti.b_row0);
            if (BN == 256) tma_load_2d(&tmB, &full[stage], sb + 128 * 128, kx, ti.b_row1);
          }
          if constexpr (MX) {
            constexpr uint32_t ab = 512u * C::SF_ATOMS;  // one stage's atoms of 128 rows, contiguous
            uint8_t *sfs = sf_base + stage * C::SF_STAGE;
            const int kg = NV ? kc >> 6 : kc >> 7;
            size_t oa = (static_cast<size_t>(a_row >> 7) * g.sfa_kg + kg) * 512;
            size_t ob0 = (static_cast<size_t>(ti.b_row0 >> 7) * g.sfb_kg + kg) * 512;
            size_t ob1 = (static_cast<size_t>(ti.b_row1 >> 7) * g.sfb_kg + kg) * 512;
            // debug builds: a scale atom past its buffer is recorded and read from offset 0
            if (!MOE_BOUNDS_OK(oa + ab <= static_cast<size_t>(g.sfa_bytes), g.status)) oa = 0;
            if (!MOE_BOUNDS_OK(ob0 + ab <= static_cast<size_t>(g.sfb_bytes), g.status)) ob0 = 0;
            if (BN == 256 && !MOE_BOUNDS_OK(ob1 + ab <= static_cast<size_t>(g.sfb_bytes), g.status)) ob1 = 0;
            bulk_load(sfs, g.sfa + oa, ab, &full[stage]);
            bulk_load(sfs + ab, g.sfb + ob0, ab, &full[stage]);
            if (BN == 256) bulk_load(sfs + 2 * ab, g.sfb + ob1, ab, &full[stage]);
          }
          if (++stage == C::STAGES) {
            stage = 0;
            ph ^= 1u;
          }
        }
      }
      // Let every copy this thread started land before the CTA exits.
      for (int s = 0; s < C::STAGES; ++s)
        if (armed[s] >= 0) {
          volatile int no_abort = 0;
          mbar_wait(&full[s], static_cast<uint32_t>(armed[s]), &no_abort, g.status, g.timeout_ns);
        }
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer
    // SF_FIRST: a tile's first scale copies go to the tensor pipe before the
    // wait for the accumulator, so they run while the epilogue still reads it.
    // Only the SwiGLU-backward GEMM gains from it (its epilogue holds the
    // accumulator longest); the other GEMMs measured slightly slower.
    constexpr bool SF_FIRST = MX && EPI == EPI_SWIGLU_BWD;
    if (lane == 0) {
      int stage = 0;
      uint32_t ph = 0;
      int acc = 0;
      uint32_t aph = 0;
      bool ok = true;
      for (int i = cta; i < total && ok; i += ncta) {
        const Tile ti = decode_tile<C::BK, BN, EPI>(g, i, il);
        if (ti.nk == 0 && g.skip_empty) continue;  // zeros written by another launch
        if (!SF_FIRST || ti.nk == 0) {
          if (!mbar_wait(&tempty[acc], aph ^ 1u, abort_flag, g.status, g.timeout_ns)) break;
          tc_fence_after();
        }
        const uint32_t dt = tmem_base + static_cast<uint32_t>(acc * BN);
        for (int kb = 0; kb < ti.nk; ++kb) {
          if (!mbar_wait(&full[stage], ph, abort_flag, g.status, g.timeout_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + stage * C::STAGE_BYTES);
          const uint32_t sb = sa + C::A_BYTES;
          const uint32_t sfa_col = tmem_base + C::SF_COL0 + stage * C::SF_COLS;
          const uint32_t sfb_col = sfa_col + C::SFA_COLS;
          if constexpr (MX) {
            constexpr uint32_t ab = 512u * C::SF_ATOMS;
            const uint32_t sfs = smem_u32(sf_base + stage * C::SF_STAGE);
#pragma unroll
            for (int a = 0; a < C::SF_ATOMS; ++a) {
              tmem_cp_32x128b_warpx4(sfa_col + 4 * a, plain_desc_sbo128(sfs + 512 * a));
#pragma unroll
              for (int c = 0; c < BN / 128; ++c)
                tmem_cp_32x128b_warpx4(sfb_col + a * (BN / 32) + 4 * c,
                                       plain_desc_sbo128(sfs + ab + ab * c + 512 * a));
            }
          }
          if (SF_FIRST && kb == 0) {
            if (!mbar_wait(&tempty[acc], aph ^ 1u, abort_flag, g.status, g.timeout_ns)) {
              ok = false;
              break;
            }
            tc_fence_after();
          }
#pragma unroll
          for (int k = 0; k < C::KSTEPS; ++k) {
            const uint64_t ad = sw128_desc(sa + 32 * k);
            const uint64_t bd = sw128_desc(sb + 32 * k);
            const uint32_t accum = (kb | k) ? 1u : 0u;
            if constexpr (NV)  // 4X: all four scale bytes of a row's word feed MMA k (scale ids 0)
              mma_nvf4(dt, ad, bd, C::IDESC, sfa_col + 4 * k, sfb_col + k * (BN / 32), accum);
            else if constexpr (MX)
              mma_mxf8(dt, ad, bd, idesc_sf_ids(C::IDESC, k, k), sfa_col, sfb_col, accum);
            else
              mma_bf16(dt, ad, bd, C::IDESC, accum);
          }
          mma_commit(&empty[stage]);
          if (++stage == C::STAGES) {
            stage = 0;
            ph ^= 1u;
          }
        }
        if (!ok) break;
        if constexpr (RING) {
          // Every load of this tile from its ring slot has landed in shared memory.
          red_release_add_gpu(g.ring.freed + (ti.a_row >> 7) % g.ring.slots, 1);
        }
        mma_commit(&tfull[acc]);
        if (++acc == C::NUM_ACC) {
          acc = 0;
          aph ^= 1u;
        }
      }
      // All MMAs this thread issued must finish before TMEM is released.
      mma_commit(done);
      volatile int no_abort = 0;
      mbar_wait(done, 0, &no_abort, g.status, g.timeout_ns);
    }
  } else {
    // ------------------------------------------------ epilogue (warps 2..)
    constexpr int NEPI = epi_warps<EPI, BN>();
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int part = (warp - 2) >> 2;  // which half of the columns (8 epilogue warps)
    const int r = q * 32 + lane;
    Stager st(staging + (warp - 2) * (C::STAGING_BYTES / NEPI));
    const OutView vO = out_view(g.out, g.ldo, g.out_rows, EPI == EPI_STORE_F32 ? 4 : 2);
    const OutView vO2 = out_view(g.out2, g.ldo2, g.out_rows, 2);
    const OutView vQ = out_view(g.outq, g.ldq, g.out_rows, 1);
    int acc = 0;
    uint32_t aph = 0;
    for (int i = cta; i < total; i += ncta) {
      const Tile ti = decode_tile<C::BK, BN, EPI>(g, i, il);
      if (ti.nk == 0 && g.skip_empty) continue;  // zeros written by another launch
      if constexpr (EPI == EPI_SWIGLU_BWD) {
        // The saved G|U rows this tile's epilogue reads come from HBM: pull them
        // into L2 while the main loop runs.
        const long prow = ti.out_row + r;
        const __nv_bfloat16 *gu = reinterpret_cast<const __nv_bfloat16 *>(g.aux) + prow * g.ld_aux;
        bulk_prefetch_l2(gu + ti.out_col, BN * 2);
        bulk_prefetch_l2(gu + g.m_half + ti.out_col, BN * 2);
      }
      if (!mbar_wait(&tfull[acc], aph, abort_flag, g.status, g.timeout_ns)) break;
      tc_fence_after();
      const uint32_t tb =
          tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * BN);
      const int row0 = ti.out_row + q * 32;  // first output row of this warp
      const long grow = ti.out_row + r;
      auto release = [&]() {
        tc_fence_before();
        mbar_arrive(&tempty[acc]);
      };
      float sc = 1.0f;  // NVFP4: the inverse of both operands' second-level scales
      if constexpr (NV) sc = 1.0f / ((g.a_gscale ? __ldg(g.a_gscale) : 1.0f) * __ldg(g.b_gscale + ti.e));
      constexpr bool STASH = EPI == EPI_SWIGLU_BWD && C::STASH;
      const uint32_t ts = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(C::STASH_COL);
      epilogue_tile_split<EPI, BN, DUMP, NV, STASH>(g, vO, vO2, vQ, st, tb, ti.nk, row0, grow, ti.out_col, lane,
                                                    part, true, release, sc, ts);
      if (++acc == C::NUM_ACC) {
        acc = 0;
        aph ^= 1u;
      }
    }
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
}

template <int F, int BN, int EPI, bool DUMP = false>
cudaError_t launch_one(const CUtensorMap &ta, const CUtensorMap &tb, const GemmArgs &g, int grid,
                       cudaStream_t s) {
  using C = Cfg<F, BN>;
  static bool attr_set = false;  // per instantiation; idempotent, benign if repeated
  if (!attr_set) {
    const cudaError_t e = cudaFuncSetAttribute(gemm_kernel<F, BN, EPI, false, DUMP>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               static_cast<int>(C::SMEM));
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  gemm_kernel<F, BN, EPI, false, DUMP><<<grid, 64 + 32 * epi_warps<EPI, BN>(), C::SMEM, s>>>(ta, tb, g);
  return cudaGetLastError();
}

int ring_ctas_query() {
  using C = Cfg<FMT_MXFP8, 256>;
  if (cudaFuncSetAttribute(gemm_kernel<FMT_MXFP8, 256, EPI_SWIGLU, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(C::SMEM)) != cudaSuccess)
    return 0;
  int per_sm = 0, dev = 0, sms = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, gemm_kernel<FMT_MXFP8, 256, EPI_SWIGLU, true>,
                                                    64 + 32 * epi_warps<EPI_SWIGLU, 256>(),
                                                    C::SMEM) != cudaSuccess ||
      cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return 0;
  return per_sm * sms;
}

int ring_ctas_resident() {
  static int memo[64] = {};
  return per_device_memo(memo, ring_ctas_query);
}

}  // namespace

int ring_max_ctas() { return ring_ctas_resident(); }

cudaError_t launch_gemm_ring(const CUtensorMap &ta, const CUtensorMap &tb, const GemmArgs &g, int grid,
                             cudaStream_t s) {
  using C = Cfg<FMT_MXFP8, 256>;
  // Gather and GEMM CTAs wait on each other: all of them must be resident at
  // once, which the cooperative launch guarantees (or refuses).
  if (grid <= g.ring.gather_ctas || g.ring.gather_ctas <= 0 || grid > ring_ctas_resident())
    return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(64 + 32 * epi_warps<EPI_SWIGLU, 256>(), 1, 1);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gemm_kernel<FMT_MXFP8, 256, EPI_SWIGLU, true>, ta, tb, g);
}

cudaError_t launch_gemm(int fmt, int bn, int epi, const CUtensorMap &ta, const CUtensorMap &tb,
                        const GemmArgs &g, int grid, cudaStream_t s) {
  if (grid <= 0) return cudaSuccess;
  if (g.dump) {  // test hook: the MXFP8 gate/up GEMM that also stores its fp32 h
    if (fmt == FMT_MXFP8 && bn == 256 && epi == EPI_SWIGLU)
      return launch_one<FMT_MXFP8, 256, EPI_SWIGLU, true>(ta, tb, g, grid, s);
    return cudaErrorInvalidValue;
  }
#define MOE_GEMM_CASE(FV, BNV, EPIV) \
  if (fmt == FV && bn == BNV && epi == EPIV) \
    return launch_one<FV, BNV, EPIV>(ta, tb, g, grid, s);
  MOE_GEMM_CASE(FMT_BF16, 256, EPI_STORE)
  MOE_GEMM_CASE(FMT_BF16, 128, EPI_STORE)
  MOE_GEMM_CASE(FMT_BF16, 256, EPI_SWIGLU)
  MOE_GEMM_CASE(FMT_BF16, 256, EPI_SWIGLU_BWD)
  MOE_GEMM_CASE(FMT_BF16, 128, EPI_SWIGLU_BWD)
  MOE_GEMM_CASE(FMT_BF16, 256, EPI_STORE_F32)
  MOE_GEMM_CASE(FMT_BF16, 128, EPI_STORE_F32)
  MOE_GEMM_CASE(FMT_BF16, 256, EPI_ADD_BF16)
  MOE_GEMM_CASE(FMT_BF16, 128, EPI_ADD_BF16)
  MOE_GEMM_CASE(FMT_MXFP8, 256, EPI_STORE)
  MOE_GEMM_CASE(FMT_MXFP8, 128, EPI_STORE)
  MOE_GEMM_CASE(FMT_MXFP8, 256, EPI_SWIGLU)
  MOE_GEMM_CASE(FMT_MXFP8, 256, EPI_SWIGLU_BWD)
  MOE_GEMM_CASE(FMT_MXFP8, 128, EPI_SWIGLU_BWD)
  MOE_GEMM_CASE(FMT_NVFP4, 256, EPI_STORE)
  MOE_GEMM_CASE(FMT_NVFP4, 128, EPI_STORE)
  MOE_GEMM_CASE(FMT_NVFP4, 256, EPI_SWIGLU)
#undef MOE_GEMM_CASE
  return cudaErrorInvalidValue;
}

}  // namespace moe
