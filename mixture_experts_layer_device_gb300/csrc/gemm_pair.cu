// Grouped expert GEMMs on CTA pairs (tcgen05 cta_group::2): the BF16 expert
// GEMMs and the shared expert, which stays in BF16 ("Mixture-of-Kittens" wiki
// page, Key claims, MXFP8 bullet).
//
// A cluster of two CTAs on two SMs computes a 256 x 256 output tile: each CTA
// loads 128 rows of A and one 128-row half of B into its own shared memory and
// owns 128 rows x 256 fp32 columns of the accumulator in its own TMEM; one
// thread of the pair leader issues the 2-CTA MMAs.  Per SM this halves the B
// bytes loaded for the same MMA work (0.75x the operand bytes per FLOP of a
// 128 x 256 single-CTA tile), which is what limits the single-CTA kernel: its
// throughput scales with operand bytes per FLOP.  Stages are 32 KB, so six fit
// where the single-CTA kernel had four 48 KB stages.
//
// Tile schedules match the single-CTA kernel (GROUP_M, DENSE, GROUP_K) with two
// consecutive 128-row M-tiles of the same expert forming one pair tile; when an
// expert has an odd number of M-tiles, the last pair's second half repeats the
// first half's rows and stores nothing.  Handoffs: the producers of both CTAs
// signal the leader's "full" mbarrier (TMA with cta_group::2); the leader's MMA
// commits multicast to the "empty" and "tfull" mbarriers of both CTAs; the
// epilogue warps of both CTAs arrive on the leader's "tempty" mbarrier.  Every
// wait is bounded (see mbar_wait).
//
// Method reference ("Mixture-of-Kittens" wiki page): expert grouped GEMMs in
// MXFP8 with fused SwiGLU and quantisation (flowchart, Key claims), SM roles
// handing off through counters rather than a global barrier (TL;DR).
#include "common.cuh"
#include "gemm_common.cuh"
#include "kernels.h"

namespace moe {

namespace {

using namespace gemm_detail;

template <bool MX, int NUM_ACC>
struct PairCfg {
  static constexpr int BN = 256;            // accumulator columns (the pair tile's N)
  static constexpr int BK = MX ? 128 : 64;  // elements per 128-byte smem row
  static constexpr int UK = MX ? 32 : 16;
  static constexpr int KSTEPS = BK / UK;
  static constexpr int A_BYTES = 128 * 128;  // this CTA's 128 rows of A
  static constexpr int B_BYTES = 128 * 128;  // this CTA's half (128 rows) of B
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int STAGES = 6;
  static constexpr int SF_STAGE = MX ? 3 * 512 : 0;  // SFA (own rows) + SFB (both halves)
  // Scale factors get their own 12 TMEM columns per pipeline stage (4 for A, 8
  // for B), so copying a stage's scales never waits for the MMAs still reading
  // the previous stage's.
  static constexpr int SF_COLS = 12;
  static constexpr int SF_COL0 = NUM_ACC * BN;
  static constexpr uint32_t TMEM_COLS = (SF_COL0 + (MX ? STAGES * SF_COLS : 0)) <= 256 ? 256 : 512;
  static constexpr uint32_t TX_BYTES = 2 * (STAGE_BYTES + SF_STAGE);  // both CTAs, on the leader
  static constexpr uint32_t IDESC = MX ? idesc_mxf8(256, BN) : idesc_bf16(256, BN);
  static constexpr int STAGING_BYTES = 4 * 4096;
  static constexpr int PAIROFF_BYTES = 4112;  // pair offsets of up to 1024 experts (16-byte multiple)
  static constexpr int NBAR = 2 * STAGES + 2 * NUM_ACC + 1;
  static constexpr size_t SMEM = 1024 + static_cast<size_t>(STAGES) * (STAGE_BYTES + SF_STAGE) +
                                 STAGING_BYTES + PAIROFF_BYTES + NBAR * 8 + 16;
  static_assert(SF_COL0 + (MX ? STAGES * SF_COLS : 0) <= 512, "TMEM columns");
  static_assert(SMEM <= 232448, "shared memory");
};

struct PairTile {
  int a_row, k0, nk, b_row0, b_row1, out_row, out_col;
  bool store;
};

MOE_DEV int pair_units(const GemmArgs &g, const int *pairoff) {
  if (g.sched == SCHED_GROUP_M) return g.n_tiles * pairoff[g.E];
  if (g.sched == SCHED_DENSE) return g.n_tiles * ((((g.M + 127) >> 7) + 1) >> 1);
  return g.E * ((g.M >> 7) >> 1) * g.n_tiles;
}

template <int BK, int EPI>
MOE_DEV PairTile decode_pair(const GemmArgs &g, const int *pairoff, int u, uint32_t rank) {
  PairTile ti;
  const int nt = g.n_tiles;
  int e = 0, ntile, m_own;
  ti.store = true;
  if (g.sched == SCHED_GROUP_M) {
    int lo = 0, hi = g.E - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (nt * pairoff[mid] <= u) lo = mid;
      else hi = mid - 1;
    }
    e = lo;
    const int local = u - nt * pairoff[e];
    const int pair = local / nt;
    ntile = local % nt;
    const int ms = __ldg(g.poff + e) >> 7;
    const int mt_e = (__ldg(g.poff + e + 1) >> 7) - ms;
    const int m_lead = ms + 2 * pair;
    m_own = m_lead + static_cast<int>(rank);
    if (2 * pair + static_cast<int>(rank) >= mt_e) {
      m_own = m_lead;
      ti.store = false;
    }
    ti.a_row = m_own * 128;
    ti.k0 = 0;
    ti.nk = g.K / BK;
    ti.out_row = ti.a_row;
  } else if (g.sched == SCHED_DENSE) {
    const int MT = (g.M + 127) >> 7;
    const int pair = u / nt;
    ntile = u % nt;
    m_own = 2 * pair + static_cast<int>(rank);
    if (m_own >= MT) {
      m_own = 2 * pair;
      ti.store = false;
    }
    ti.a_row = m_own * 128;
    ti.k0 = 0;
    ti.nk = g.K / BK;
    ti.out_row = ti.a_row;
  } else {
    const int per = ((g.M >> 7) >> 1) * nt;
    e = u / per;
    const int r = u % per;
    const int pair = r / nt;
    ntile = r % nt;
    m_own = 2 * pair + static_cast<int>(rank);
    ti.a_row = m_own * 128;
    if (g.poff) {
      ti.k0 = __ldg(g.poff + e);
      ti.nk = (__ldg(g.poff + e + 1) - ti.k0) / BK;
    } else {
      ti.k0 = 0;
      ti.nk = g.K / BK;
    }
    ti.out_row = e * g.M + ti.a_row;
  }
  if (EPI == EPI_SWIGLU) {
    ti.b_row0 = e * g.b_rows_per_group + ntile * 128;  // gate rows -> leader
    ti.b_row1 = ti.b_row0 + g.b_split;                   // up rows   -> follower
    ti.out_col = ntile * 128;
  } else {
    ti.b_row0 = (g.sched == SCHED_GROUP_K ? 0 : e * g.b_rows_per_group) + ntile * 256;
    ti.b_row1 = ti.b_row0 + 128;
    ti.out_col = ntile * 256;
  }
  return ti;
}

template <bool MX, int EPI, int NUM_ACC>
__global__ void __launch_bounds__(192, 1)
    gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const __grid_constant__ CUtensorMap tmSFA,
                     const __grid_constant__ CUtensorMap tmSFB, const GemmArgs g) {
  using C = PairCfg<MX, NUM_ACC>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  uint8_t *sf_base = smem + C::STAGES * C::STAGE_BYTES;
  uint8_t *staging = sf_base + C::STAGES * C::SF_STAGE;
  int *pairoff = reinterpret_cast<int *>(staging + C::STAGING_BYTES);
  uint64_t *bars = reinterpret_cast<uint64_t *>(reinterpret_cast<uint8_t *>(pairoff) + C::PAIROFF_BYTES);
  uint64_t *full = bars;
  uint64_t *empty = bars + C::STAGES;
  uint64_t *tfull = bars + 2 * C::STAGES;
  uint64_t *tempty = tfull + NUM_ACC;
  uint64_t *done = tempty + NUM_ACC;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(done + 1);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const bool leader = rank == 0;
  const int cluster_id = blockIdx.x >> 1;
  const int num_clusters = gridDim.x >> 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < NUM_ACC; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 256);  // epilogue threads of both CTAs
    }
    mbar_init(done, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (g.sched == SCHED_GROUP_M && warp == 0) {
    // pairoff[e] = sum over e' < e of ceil(m-tiles of e' / 2)
    int run = 0;
    for (int base = 0; base < g.E; base += 32) {
      const int e = base + lane;
      int c = 0;
      if (e < g.E) c = ((__ldg(g.poff + e + 1) >> 7) - (__ldg(g.poff + e) >> 7) + 1) >> 1;
      int inc = c;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, inc, off);
        if (lane >= off) inc += o;
      }
      if (e < g.E) pairoff[e] = run + inc - c;
      run += __shfl_sync(0xffffffffu, inc, 31);
    }
    if (lane == 0) pairoff[g.E] = run;
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, C::TMEM_COLS);
    tmem_relinquish_pair();
    tc_fence_before();
  }
  __syncthreads();
  cluster_sync();  // both CTAs' barriers exist before any cross-CTA signal
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int total = pair_units(g, pairoff);

  if (warp == 0) {
    // ------------------------------------------------ TMA producer (both CTAs)
    if (lane == 0) {
      prefetch_tensormap(&tmA);
      prefetch_tensormap(&tmB);
      int stage = 0;
      uint32_t ph = 0;
      for (int u = cluster_id; u < total && !*abort_flag && !g.debug_starve; u += num_clusters) {
        const PairTile ti = decode_pair<C::BK, EPI>(g, pairoff, u, rank);
        const int b_row = leader ? ti.b_row0 : ti.b_row1;
        for (int kb = 0; kb < ti.nk; ++kb) {
          if (!mbar_wait(&empty[stage], ph ^ 1u, abort_flag, g.status, g.timeout_ns)) break;
          uint8_t *sa = smem + stage * C::STAGE_BYTES;
          uint8_t *sb = sa + C::A_BYTES;
          if (leader) mbar_arrive_expect_tx(&full[stage], C::TX_BYTES);
          const uint32_t lead_full = peer_smem(smem_u32(&full[stage]), 0);
          const int kc = ti.k0 + kb * C::BK;
          tma_load_2d_pair(&tmA, lead_full, sa, kc, ti.a_row);
          tma_load_2d_pair(&tmB, lead_full, sb, kc, b_row);
          if constexpr (MX) {
            // 512-byte scale atoms, each two 256-byte rows of the 2-D scale maps
            uint8_t *sfs = sf_base + stage * C::SF_STAGE;
            const int kg = kc >> 7;
            tma_load_2d_pair(&tmSFA, lead_full, sfs, 0, 2 * ((ti.a_row >> 7) * g.sfa_kg + kg));
            tma_load_2d_pair(&tmSFB, lead_full, sfs + 512, 0, 2 * ((ti.b_row0 >> 7) * g.sfb_kg + kg));
            tma_load_2d_pair(&tmSFB, lead_full, sfs + 1024, 0, 2 * ((ti.b_row1 >> 7) * g.sfb_kg + kg));
          }
          if (++stage == C::STAGES) {
            stage = 0;
            ph ^= 1u;
          }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer (pair leader)
    if (leader && lane == 0) {
      int stage = 0;
      uint32_t ph = 0;
      int acc = 0;
      uint32_t aph = 0;
      bool ok = true;
      for (int u = cluster_id; u < total && ok; u += num_clusters) {
        const PairTile ti = decode_pair<C::BK, EPI>(g, pairoff, u, rank);
        if (!mbar_wait(&tempty[acc], aph ^ 1u, abort_flag, g.status, g.timeout_ns)) break;
        tc_fence_after();
        const uint32_t dt = tmem_base + static_cast<uint32_t>(acc * C::BN);
        for (int kb = 0; kb < ti.nk; ++kb) {
          if (!mbar_wait(&full[stage], ph, abort_flag, g.status, g.timeout_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + stage * C::STAGE_BYTES);
          const uint32_t sb = sa + C::A_BYTES;
          const uint32_t sfa_col = tmem_base + C::SF_COL0 + stage * C::SF_COLS;
          const uint32_t sfb_col = sfa_col + 4;
          if constexpr (MX) {
            const uint32_t sfs = smem_u32(sf_base + stage * C::SF_STAGE);
            tmem_cp_pair_32x128b_warpx4(sfa_col, plain_desc_sbo128(sfs));
            tmem_cp_pair_32x128b_warpx4(sfb_col, plain_desc_sbo128(sfs + 512));
            tmem_cp_pair_32x128b_warpx4(sfb_col + 4, plain_desc_sbo128(sfs + 1024));
          }
#pragma unroll
          for (int k = 0; k < C::KSTEPS; ++k) {
            const uint64_t ad = sw128_desc(sa + 32 * k);
            const uint64_t bd = sw128_desc(sb + 32 * k);
            const uint32_t accum = (kb | k) ? 1u : 0u;
            if constexpr (MX)
              mma_mxf8_pair(dt, ad, bd, idesc_sf_ids(C::IDESC, k, k), sfa_col, sfb_col, accum);
            else
              mma_bf16_pair(dt, ad, bd, C::IDESC, accum);
          }
          mma_commit_pair_mc(&empty[stage], 3);
          if (++stage == C::STAGES) {
            stage = 0;
            ph ^= 1u;
          }
        }
        if (!ok) break;
        mma_commit_pair_mc(&tfull[acc], 3);
        if (++acc == NUM_ACC) {
          acc = 0;
          aph ^= 1u;
        }
      }
      mma_commit_pair_mc(done, 1);
      volatile int no_abort = 0;
      mbar_wait(done, 0, &no_abort, g.status, g.timeout_ns);
    }
  } else {
    // ------------------------------------------------ epilogue (warps 2..5, both CTAs)
    const int q = warp & 3;
    const int r = q * 32 + lane;
    Stager st(staging + (warp - 2) * 4096);
    const OutView vO = out_view(g.out, g.ldo, g.out_rows, 2);
    const OutView vO2 = out_view(g.out2, g.ldo2, g.out_rows, 2);
    const OutView vQ = out_view(g.outq, g.ldq, g.out_rows, 1);
    int acc = 0;
    uint32_t aph = 0;
    for (int u = cluster_id; u < total; u += num_clusters) {
      const PairTile ti = decode_pair<C::BK, EPI>(g, pairoff, u, rank);
      if constexpr (EPI == EPI_SWIGLU_BWD) {
        if (ti.store) {
          const __nv_bfloat16 *gu =
              reinterpret_cast<const __nv_bfloat16 *>(g.aux) + (ti.out_row + r) * g.ld_aux;
          bulk_prefetch_l2(gu + ti.out_col, C::BN * 2);
          bulk_prefetch_l2(gu + g.m_half + ti.out_col, C::BN * 2);
        }
      }
      if (!mbar_wait(&tfull[acc], aph, abort_flag, g.status, g.timeout_ns)) break;
      tc_fence_after();
      const uint32_t tb =
          tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * C::BN);
      const int row0 = ti.out_row + q * 32;
      const long grow = ti.out_row + r;
      const uint32_t tempty_addr = smem_u32(&tempty[acc]);
      auto release = [&]() {
        tc_fence_before();
        if (leader) mbar_arrive(&tempty[acc]);
        else mbar_arrive_remote(peer_smem(tempty_addr, 0));
      };
      epilogue_tile<EPI, C::BN>(g, vO, vO2, vQ, st, tb, ti.nk, row0, grow, ti.out_col, lane,
                                ti.store, release);
      if (++acc == NUM_ACC) {
        acc = 0;
        aph ^= 1u;
      }
    }
  }

  __syncthreads();
  cluster_sync();  // no CTA leaves while its peer may still signal it
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, C::TMEM_COLS);
  }
}

template <bool MX, int EPI, int NUM_ACC>
cudaError_t launch_pair_one(const PairMaps &m, const GemmArgs &g, int clusters, cudaStream_t s) {
  using C = PairCfg<MX, NUM_ACC>;
  static bool attr_set = false;
  if (!attr_set) {
    const cudaError_t e = cudaFuncSetAttribute(gemm_pair_kernel<MX, EPI, NUM_ACC>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               static_cast<int>(C::SMEM));
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * clusters, 1, 1);
  cfg.blockDim = dim3(192, 1, 1);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gemm_pair_kernel<MX, EPI, NUM_ACC>, m.a, m.b, m.sfa, m.sfb, g);
}

}  // namespace

cudaError_t launch_gemm_pair(bool mx, int epi, const PairMaps &m, const GemmArgs &g, int clusters,
                             cudaStream_t s) {
  if (clusters <= 0) return cudaSuccess;
  // BF16 with two accumulators (2 x 256 TMEM columns).  The kernel template
  // also supports MXFP8 (block-scaled MMA with scale copies per stage, one
  // accumulator); it measured slower than the single-CTA MXFP8 kernel, so it is
  // not instantiated.
#define MOE_PAIR_CASE(MXV, EPIV, NA) \
  if (mx == MXV && epi == EPIV) return launch_pair_one<MXV, EPIV, NA>(m, g, clusters, s);
  MOE_PAIR_CASE(false, EPI_STORE, 2)
  MOE_PAIR_CASE(false, EPI_SWIGLU, 2)
  MOE_PAIR_CASE(false, EPI_SWIGLU_BWD, 2)
#undef MOE_PAIR_CASE
  return cudaErrorInvalidValue;
}

namespace {
template <bool MX, int EPI, int NUM_ACC>
int max_clusters_one_query() {
  using C = PairCfg<MX, NUM_ACC>;
  if (cudaFuncSetAttribute(gemm_pair_kernel<MX, EPI, NUM_ACC>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(C::SMEM)) != cudaSuccess)
    return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2, 1, 1);
  cfg.blockDim = dim3(192, 1, 1);
  cfg.dynamicSmemBytes = C::SMEM;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, gemm_pair_kernel<MX, EPI, NUM_ACC>, &cfg) != cudaSuccess) return 0;
  return n;
}
template <bool MX, int EPI, int NUM_ACC>
int max_clusters_one() {
  static int memo[64] = {};
  return per_device_memo(memo, max_clusters_one_query<MX, EPI, NUM_ACC>);
}
}  // namespace

// Number of CTA pairs of the pair kernel that are resident at once (0 on error).
int pair_max_clusters(bool mx, int epi) {
#define MOE_PAIR_OCC(MXV, EPIV, NA) \
  if (mx == MXV && epi == EPIV) return max_clusters_one<MXV, EPIV, NA>();
  MOE_PAIR_OCC(false, EPI_STORE, 2)
  MOE_PAIR_OCC(false, EPI_SWIGLU, 2)
  MOE_PAIR_OCC(false, EPI_SWIGLU_BWD, 2)
#undef MOE_PAIR_OCC
  return 0;
}

}  // namespace moe
