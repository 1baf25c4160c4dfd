// Host side of the C ABI declared in include/moe.h: argument checks, the
// layout of the caller-owned workspace / saved buffers, TMA tensor maps, and
// the launch sequence of the forward and backward passes.  Nothing here
// allocates memory or synchronises the host with the device (except
// moe_get_status, which exists to do exactly that).
//
// The launch sequence follows the method's pipeline ("Mixture-of-Kittens" wiki
// page, flowchart): route, device-side schedule, dispatch with fused MXFP8
// quantisation, expert grouped GEMMs with fused SwiGLU, fixed-order combine,
// the BF16 shared expert (Key claims, MXFP8 bullet); the backward runs the
// reverse combine first and the reverse dispatch last (Key claims,
// communication-direction bullet).
#include <cuda.h>
#include <cuda_runtime.h>
#include <string.h>

#include <mutex>

#include "../../include/moe.h"
#include "kernels.h"

namespace {

using moe::GemmArgs;
using moe::RouteBufs;

// ---------------------------------------------------------------- shapes
// Gather CTAs of the ring kernel when moe_config.gather_sms is 0.
constexpr int kDefaultGatherCtas = 8;

struct Dims {
  int T, d, m, E, k, ms;
  bool mx, bwd, starve;
  bool nv;             // NVFP4 experts (forward only)
  bool dump;           // MOE_FLAG_DEBUG_DUMP with MXFP8 experts
  bool ring;           // MXFP8 forward dispatch through the persistent ring kernel
  float aux_alpha;     // load-balancing term weight (0 = none)
  int ring_slots;      // ring capacity in 128-row tiles
  int gather_ctas;     // gather CTAs of the ring kernel
  long R, Rp, Tp;
  int nchunks;
};

int check_config(const moe_config *c, Dims *D) {
  if (!c) return MOE_ERR_ARG;
  if (c->T <= 0 || c->d <= 0 || c->m <= 0 || c->E <= 0 || c->k <= 0 || c->m_shared < 0)
    return MOE_ERR_ARG;
  if (c->k > c->E || c->k > 16 || c->E > 1024) return MOE_ERR_SHAPE;
  if (c->dtype != MOE_BF16 && c->dtype != MOE_MXFP8 && c->dtype != MOE_NVFP4) return MOE_ERR_ARG;
  if (c->dtype == MOE_NVFP4 && (c->flags & MOE_FLAG_BACKWARD)) return MOE_ERR_ARG;  // forward only
  if (c->dtype == MOE_NVFP4 && c->m % 256) return MOE_ERR_SHAPE;  // 256-deep stages along K = m
  if ((c->flags & ~(MOE_FLAG_BACKWARD | MOE_FLAG_DEBUG_STARVE | MOE_FLAG_DEBUG_DUMP)) != 0) return MOE_ERR_ARG;
  if (c->d % 256 || c->m % 128 || c->m_shared % 128) return MOE_ERR_SHAPE;
  if (c->ring_rows < 0 || c->gather_sms < 0 || c->gather_sms > 64) return MOE_ERR_ARG;
  if (c->ring_rows > 0 && c->dtype != MOE_MXFP8) return MOE_ERR_ARG;
  if (c->ring_rows % 128) return MOE_ERR_SHAPE;
  if (c->ring_rows > 0 && c->d > 8192) return MOE_ERR_SHAPE;  // the ring's gather copies whole rows
  if (c->ring_rows > 0 && (c->flags & MOE_FLAG_DEBUG_DUMP)) return MOE_ERR_ARG;  // no dump in the ring launch
  if (!(c->aux_alpha >= 0.0f) || !(c->aux_alpha < 1e30f)) return MOE_ERR_ARG;  // finite, non-negative
  const long R = static_cast<long>(c->T) * c->k;
  const long Rp = (R + 127L * c->E + 127) / 128 * 128;
  if (Rp >= (1L << 31)) return MOE_ERR_SHAPE;
  D->T = c->T;
  D->d = c->d;
  D->m = c->m;
  D->E = c->E;
  D->k = c->k;
  D->ms = c->m_shared;
  D->mx = c->dtype == MOE_MXFP8;
  D->nv = c->dtype == MOE_NVFP4;
  D->bwd = (c->flags & MOE_FLAG_BACKWARD) != 0;
  D->starve = (c->flags & MOE_FLAG_DEBUG_STARVE) != 0;
  D->dump = D->mx && (c->flags & MOE_FLAG_DEBUG_DUMP) != 0;
  D->ring = c->ring_rows > 0;
  D->aux_alpha = c->aux_alpha;
  D->ring_slots = c->ring_rows / 128;
  D->gather_ctas = c->gather_sms > 0 ? c->gather_sms : kDefaultGatherCtas;
  D->R = R;
  D->Rp = Rp;
  D->Tp = (c->T + 127L) / 128 * 128;
  D->nchunks = static_cast<int>((R + moe::kSchedChunk - 1) / moe::kSchedChunk);
  return MOE_OK;
}

// ---------------------------------------------------------------- layouts
struct Entry {
  const char *name;
  size_t off, bytes;
};
struct Layout {
  Entry e[80];
  int n = 0;
  size_t total = 0;
  void add(const char *name, size_t bytes) {
    if (bytes == 0) return;
    const size_t off = (total + 255) & ~static_cast<size_t>(255);
    e[n++] = {name, off, bytes};
    total = off + bytes;
  }
  const Entry *find(const char *name) const {
    for (int i = 0; i < n; ++i)
      if (strcmp(e[i].name, name) == 0) return &e[i];
    return nullptr;
  }
  char *ptr(void *base, const char *name) const {
    const Entry *x = find(name);
    return x ? static_cast<char *>(base) + x->off : nullptr;
  }
};

void add_route(const Dims &D, Layout &L) {
  L.add("idx", D.R * 4);
  L.add("w", D.R * 4);
  L.add("counts", D.E * 4);
  L.add("offsets", (D.E + 1) * 4);
  L.add("perm", D.R * 4);
  L.add("inv", D.R * 4);
  L.add("poff", (D.E + 1) * 4);
}

// Activations a training forward keeps for the backward.
void saved_layout(const Dims &D, Layout &L) {
  add_route(D, L);
  L.add("o", D.Rp * D.d * 2);
  L.add("GU", D.Rp * 2 * D.m * 2);
  if (D.mx) {
    // column-blocked codes of the gathered x (written by the dispatch) and of
    // h (written by the gate/up GEMM's epilogue): the wgrad operands
    L.add("xT", D.d * D.Rp);
    L.add("xT_sf", D.d * D.Rp / 32);
    L.add("hT", D.m * D.Rp);
    L.add("hT_sf", D.m * D.Rp / 32);
  } else {
    L.add("h", D.Rp * D.m * 2);
  }
  if (D.ms) {
    L.add("s_GU", D.Tp * 2 * D.ms * 2);
    L.add("s_h", D.Tp * D.ms * 2);
  }
  if (D.aux_alpha > 0.f) L.add("aux_grad", static_cast<size_t>(D.T) * D.E * 4);  // dL/dlogits
}

void ws_layout(const Dims &D, Layout &L) {
  L.add("status", 16);
  L.add("hist", static_cast<size_t>(D.nchunks) * D.E * 4);
  L.add("tile_order", static_cast<size_t>(D.Rp / 32) * 4);
  if (D.aux_alpha > 0.f) {
    L.add("aux", (1 + 2 * static_cast<size_t>(D.E)) * 4);  // [L, P[E], f[E]]
    L.add("aux_part", static_cast<size_t>(moe::balance_blocks(D.T)) * D.E * 4);
  }
  // router projection: its logits before cropping, [Tp, E rounded up to 128] fp32
  const size_t Ep = (static_cast<size_t>(D.E) + 127) / 128 * 128;
  L.add("router_lpad", static_cast<size_t>(D.Tp) * Ep * 4);
  add_route(D, L);  // used when the forward saves nothing
  const size_t eb = D.mx ? 1 : 2;
  if (D.nv) {
    // NVFP4: x's second-level scale, every token's packed codes (canonical
    // scales), the dispatched rows and h (packed codes, tiled scales)
    L.add("x_gscale", 16);
    L.add("xq", static_cast<size_t>(D.T) * D.d / 2);
    L.add("xq_sf", static_cast<size_t>(D.T) * D.d / 16);
    L.add("xs", D.Rp * D.d / 2);
    L.add("xs_sf", D.Rp * D.d / 16);
    L.add("hq", D.Rp * D.m / 2);
    L.add("hq_sf", D.Rp * D.m / 16);
  } else if (D.mx) {  // row-blocked codes of every token (the dispatch copies them per routed row)
    L.add("xq", static_cast<size_t>(D.T) * D.d);
    L.add("xq_sf", static_cast<size_t>(D.T) * D.d / 32);
  }
  if (D.nv) {
  } else if (D.ring) {  // a fixed ring of 128-row tiles instead of every dispatched row
    L.add("ring", static_cast<size_t>(D.ring_slots) * 128 * D.d);
    L.add("ring_sf", static_cast<size_t>(D.ring_slots) * 128 * D.d / 32);
    L.add("ring_ctrl", (2 * static_cast<size_t>(D.ring_slots) + 1) * 4);
  } else {
    L.add("xs", D.Rp * D.d * eb);
  }
  if (D.nv) {
  } else if (D.mx) {
    if (!D.ring) L.add("xs_sf", D.Rp * D.d / 32);
    L.add("hq", D.Rp * D.m);
    L.add("hq_sf", D.Rp * D.m / 32);
  } else {
    L.add("h", D.Rp * D.m * 2);
  }
  L.add("o", D.Rp * D.d * 2);
  if (D.ms) {
    L.add("s_h", D.Tp * D.ms * 2);
    L.add("s_out", D.Tp * D.d * 2);
  }
  if (D.dump) L.add("h_dump", D.Rp * D.m * 4);  // fp32 h before its quantisation (test hook)
  if (!D.bwd) return;
  if (D.dump) L.add("dGU_dump", D.Rp * 2 * D.m * 2);  // bf16 dG|dU before their quantisation
  // router backward: bf16 dlogits [Tp, Ep], its transpose, W_r^T [d, Ep], x^T [d, Tp] (zero-padded)
  L.add("router_g", static_cast<size_t>(D.Tp) * Ep * 2);
  L.add("router_gT", Ep * static_cast<size_t>(D.Tp) * 2);
  L.add("router_WrT", static_cast<size_t>(D.d) * Ep * 2);
  L.add("router_xT", static_cast<size_t>(D.d) * D.Tp * 2);
  L.add("g", D.R * 4);
  if (!D.mx) L.add("dO", D.Rp * D.d * 2);  // MXFP8 keeps dO only as codes
  if (!D.mx) L.add("dGU", D.Rp * 2 * D.m * 2);  // MXFP8 keeps dGU only as codes
  L.add("dX", D.Rp * D.d * 2);
  L.add("dOT", D.d * D.Rp * eb);
  if (!D.mx) L.add("hT", D.m * D.Rp * eb);  // MXFP8: kept in `saved` by the gate/up GEMM
  L.add("dGUT", 2 * D.m * D.Rp * eb);
  if (!D.mx) L.add("xT", D.d * D.Rp * eb);  // MXFP8: kept in `saved` by the dispatch
  if (D.mx) {
    L.add("dOq", D.Rp * D.d);
    L.add("dOq_sf", D.Rp * D.d / 32);
    L.add("dGUq", D.Rp * 2 * D.m);
    L.add("dGUq_sf", D.Rp * 2 * D.m / 32);
    L.add("dOT_sf", D.d * D.Rp / 32);
    L.add("dGUT_sf", 2 * D.m * D.Rp / 32);
  }
  if (D.ms) {
    L.add("s_dGU", D.Tp * 2 * D.ms * 2);
    L.add("s_dx", D.Tp * D.d * 2);
    L.add("s_dyT", D.d * D.Tp * 2);
    L.add("s_hT", D.ms * D.Tp * 2);
    L.add("s_dGUT", 2 * D.ms * D.Tp * 2);
    L.add("s_xT", D.d * D.Tp * 2);
  }
}

// ---------------------------------------------------------------- device info
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

struct DeviceInfo {
  bool ok = false;
  int num_sms = 0;
};
std::mutex g_mu;
EncodeTiledFn g_encode = nullptr;
DeviceInfo g_dev[64];

int device_info(DeviceInfo *out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MOE_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_encode) {
    cudaDriverEntryPointQueryResult q;
    void *fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn)
      return MOE_ERR_CUDA;
    g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  }
  if (!g_dev[dev].ok) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return MOE_ERR_CUDA;
    if (major != 10 || minor != 3) return MOE_ERR_DEVICE;
    g_dev[dev].num_sms = sms;
    g_dev[dev].ok = true;
  }
  *out = g_dev[dev];
  return MOE_OK;
}

// 2-D K-major tensor map: `rows` rows of `inner` elements (bf16 or 1-byte codes),
// box 128 rows x 128 bytes, 128-byte swizzle, zero fill out of bounds.
bool make_map(CUtensorMap *m, const void *base, bool bytes1, uint64_t inner, uint64_t rows) {
  const uint64_t esz = bytes1 ? 1 : 2;
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {inner * esz};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(128 / esz), 128};
  cuuint32_t estr[2] = {1, 1};
  const CUresult r = g_encode(m, bytes1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                              2, const_cast<void *>(base), dims, strides, box, estr,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// ---------------------------------------------------------------- tracing
struct Trace {
  int capacity = 0, count = 0;
  cudaEvent_t *start = nullptr, *end = nullptr;
  const char **name = nullptr;
} g_trace;

void trace_free() {
  for (int i = 0; i < g_trace.capacity; ++i) {
    cudaEventDestroy(g_trace.start[i]);
    cudaEventDestroy(g_trace.end[i]);
  }
  delete[] g_trace.start;
  delete[] g_trace.end;
  delete[] g_trace.name;
  g_trace = Trace();
}

// Brackets one launch with an event pair when tracing is enabled.
struct Traced {
  int slot = -1;
  cudaStream_t s;
  Traced(const char *name, cudaStream_t st) : s(st) {
    if (g_trace.count < g_trace.capacity) {
      slot = g_trace.count++;
      g_trace.name[slot] = name;
      cudaEventRecord(g_trace.start[slot], s);
    }
  }
  ~Traced() {
    if (slot >= 0) cudaEventRecord(g_trace.end[slot], s);
  }
};

int cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

// One GEMM launch: A [a_rows, K] and B [b_rows, K] (K-major) plus arguments;
// the outputs (g.out / out2 / outq) have out_rows rows.
struct Gemm {
  bool mx;          // block-scaled byte operands (MXFP8, or NVFP4 with nv)
  bool nv = false;  // NVFP4: packed E2M1 codes, K / 2 bytes per row
  int bn, epi;
  const void *a;
  long a_rows;
  const void *b;
  long b_rows;
  long K;
  GemmArgs g;
  long max_tiles;
  long out_rows;
  // weight gradients: the empty experts' all-zero dW, written by a plain
  // store kernel inside the same traced region (single-CTA path only)
  void *zero_dst = nullptr;
  long zero_expert_bytes = 0;
  const int *zero_counts = nullptr;
};

// 2-D view of a tiled MXFP8 scale buffer as rows of 256 bytes (box: one
// 512-byte atom = 2 rows), for the pair kernel's TMA scale loads.
bool make_sf_map(CUtensorMap *m, const void *base, uint64_t bytes) {
  cuuint64_t dims[2] = {256, bytes / 256};
  cuuint64_t strides[1] = {256};
  cuuint32_t box[2] = {256, 2};
  cuuint32_t estr[2] = {1, 1};
  return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Whether a GEMM runs on CTA pairs: BF16 with 256-wide N tiles (and, for
// weight gradients, an even number of 128-row M tiles per expert).  MXFP8
// stays on single-CTA tiles: there a 128 x 256 tile already runs the SM's
// shared-memory traffic (TMA writes + MMA operand reads) near its limit, and
// the pair's cross-SM coupling measured slower.
bool use_pair(const Gemm &q) { return q.bn == 256 && !q.mx; }

int run_pair(const Gemm &q, const DeviceInfo &dev, cudaStream_t s) {
  moe::PairMaps m;
  memset(&m, 0, sizeof(m));
  if (!make_map(&m.a, q.a, q.mx, q.K, q.a_rows) || !make_map(&m.b, q.b, q.mx, q.K, q.b_rows))
    return MOE_ERR_CUDA;
  if (q.mx && (!make_sf_map(&m.sfa, q.g.sfa, static_cast<uint64_t>(q.a_rows) * q.K / 32) ||
               !make_sf_map(&m.sfb, q.g.sfb, static_cast<uint64_t>(q.b_rows) * q.K / 32)))
    return MOE_ERR_CUDA;
  const int maxc = moe::pair_max_clusters(q.mx, q.epi);
  if (maxc <= 0) return MOE_ERR_CUDA;
  const long pairs = (q.max_tiles + 1) / 2;
  const long clusters = pairs < maxc ? pairs : maxc;
  (void)dev;
  moe::GemmArgs g = q.g;
  g.out_rows = q.out_rows;
  return cuda_status(moe::launch_gemm_pair(q.mx, q.epi, m, g, static_cast<int>(clusters), s));
}

int gemm_fmt(const Gemm &q) { return q.nv ? moe::FMT_NVFP4 : (q.mx ? moe::FMT_MXFP8 : moe::FMT_BF16); }
// The GEMM's arguments with the output rows and the scale buffers' sizes (the
// latter for the bounds checks of debug builds).
moe::GemmArgs launch_args(const Gemm &q) {
  moe::GemmArgs g = q.g;
  g.out_rows = q.out_rows;
  const long blk = q.nv ? 16 : 32;
  g.sfa_bytes = (q.a_rows + 127) / 128 * 128 * q.K / blk;
  g.sfb_bytes = (q.b_rows + 127) / 128 * 128 * q.K / blk;
  return g;
}
// Elements of the tensor maps' inner dimension: NVFP4 rows hold two codes per byte.
uint64_t map_inner(const Gemm &q) { return q.nv ? q.K / 2 : q.K; }

int run_gemm(const char *name, const Gemm &q, const DeviceInfo &dev, cudaStream_t s) {
  Traced tr(name, s);
  if (use_pair(q) && (q.g.sched != moe::SCHED_GROUP_K || (q.g.M / 128) % 2 == 0)) return run_pair(q, dev, s);
  CUtensorMap tb;
  if (!make_map(&tb, q.b, q.mx, map_inner(q), q.b_rows)) return MOE_ERR_CUDA;
  moe::GemmArgs g = launch_args(q);
  if (q.zero_dst) {
    const int rc = cuda_status(moe::launch_zero_empty_experts(q.zero_dst, q.g.E, q.zero_expert_bytes,
                                                              q.zero_counts, s));
    if (rc != MOE_OK) return rc;
    g.skip_empty = 1;
  }
  CUtensorMap ta;
  if (!make_map(&ta, q.a, q.mx, map_inner(q), q.a_rows)) return MOE_ERR_CUDA;
  const long grid = q.max_tiles < dev.num_sms ? q.max_tiles : dev.num_sms;
  return cuda_status(moe::launch_gemm(gemm_fmt(q), q.bn, q.epi, ta, tb, g, static_cast<int>(grid), s));
}

// A GEMM on the single-CTA kernel (the router's fp32-store and add-into-bf16
// epilogues exist only there); untraced, inside its caller's traced region.
int run_gemm_single(const Gemm &q, const DeviceInfo &dev, cudaStream_t s) {
  CUtensorMap ta, tb;
  if (!make_map(&ta, q.a, q.mx, q.K, q.a_rows) || !make_map(&tb, q.b, q.mx, q.K, q.b_rows)) return MOE_ERR_CUDA;
  moe::GemmArgs g = launch_args(q);
  const long grid = q.max_tiles < dev.num_sms ? q.max_tiles : dev.num_sms;
  return cuda_status(moe::launch_gemm(gemm_fmt(q), q.bn, q.epi, ta, tb, g, static_cast<int>(grid), s));
}

// The persistent ring launch: one CTA per SM, the first gather_ctas of which
// gather into the ring (fewer if the device has few SMs).
int run_gemm_ring(const char *name, const Gemm &q, const Dims &D, const DeviceInfo &dev, cudaStream_t s) {
  Traced tr(name, s);
  CUtensorMap ta, tb;
  if (!make_map(&ta, q.a, true, q.K, q.a_rows) || !make_map(&tb, q.b, true, q.K, q.b_rows)) return MOE_ERR_CUDA;
  int grid = moe::ring_max_ctas();
  if (grid > dev.num_sms) grid = dev.num_sms;
  if (grid < 2) return MOE_ERR_CUDA;
  moe::GemmArgs g = launch_args(q);
  g.ring.gather_ctas = D.gather_ctas < grid ? D.gather_ctas : grid / 2;
  return cuda_status(moe::launch_gemm_ring(ta, tb, g, grid, s));
}

int bn_for(long n) { return n % 256 == 0 ? 256 : 128; }

struct Ptrs {
  RouteBufs rb;
  int *status;
};

Ptrs route_ptrs(const Dims &D, const Layout &L, void *base, void *ws, const Layout &W) {
  Ptrs p;
  p.rb.idx = reinterpret_cast<int *>(L.ptr(base, "idx"));
  p.rb.w = reinterpret_cast<float *>(L.ptr(base, "w"));
  p.rb.counts = reinterpret_cast<int *>(L.ptr(base, "counts"));
  p.rb.offsets = reinterpret_cast<int *>(L.ptr(base, "offsets"));
  p.rb.perm = reinterpret_cast<int *>(L.ptr(base, "perm"));
  p.rb.inv = reinterpret_cast<int *>(L.ptr(base, "inv"));
  p.rb.poff = reinterpret_cast<int *>(L.ptr(base, "poff"));
  p.rb.hist = reinterpret_cast<int *>(W.ptr(ws, "hist"));
  p.rb.tile_order = reinterpret_cast<int *>(W.ptr(ws, "tile_order"));
  p.status = reinterpret_cast<int *>(W.ptr(ws, "status"));
  p.rb.n_tok = D.T;
  p.rb.n_slots = D.R;
  p.rb.n_rows = D.Rp;
  p.rb.status = p.status;
  return p;
}

GemmArgs base_args(int sched, int E, const int *poff, int *status) {
  GemmArgs g;
  memset(&g, 0, sizeof(g));
  g.sched = sched;
  g.E = E;
  g.poff = poff;
  g.status = status;
  g.timeout_ns = moe::kWaitTimeoutNs;
  return g;
}

// MOE_FLAG_DEBUG_STARVE: the gate/up GEMM's producer issues no loads and every
// wait of that launch gives up after 50 ms.
constexpr unsigned long long kStarveTimeoutNs = 50000000ull;

}  // namespace

extern "C" {

size_t moe_workspace_bytes(const moe_config *cfg) {
  Dims D;
  if (check_config(cfg, &D) != MOE_OK) return 0;
  Layout L;
  ws_layout(D, L);
  return L.total;
}

size_t moe_saved_bytes(const moe_config *cfg) {
  Dims D;
  if (check_config(cfg, &D) != MOE_OK) return 0;
  Layout L;
  saved_layout(D, L);
  return L.total;
}

int moe_buffer_info(const moe_config *cfg, int which, const char *name, size_t *offset,
                    size_t *bytes) {
  Dims D;
  const int rc = check_config(cfg, &D);
  if (rc != MOE_OK) return rc;
  if (!name || !offset || !bytes || (which != 0 && which != 1)) return MOE_ERR_ARG;
  Layout L;
  if (which == 0) saved_layout(D, L);
  else ws_layout(D, L);
  const Entry *e = L.find(name);
  if (!e) return MOE_ERR_ARG;
  *offset = e->off;
  *bytes = e->bytes;
  return MOE_OK;
}

int64_t moe_padded_rows(const moe_config *cfg) {
  Dims D;
  if (check_config(cfg, &D) != MOE_OK) return 0;
  return D.Rp;
}

int moe_quantize_mx(const void *src, int batch, int rows, int cols, int transpose, void *codes,
                    void *scales, moe_stream_t stream) {
  if (!src || !codes || !scales || batch <= 0 || rows <= 0 || cols <= 0) return MOE_ERR_ARG;
  if (rows % 128 || cols % 128) return MOE_ERR_SHAPE;
  if (!aligned16(src) || !aligned16(codes) || !aligned16(scales)) return MOE_ERR_ALIGN;
  DeviceInfo dev;
  const int rc = device_info(&dev);
  if (rc != MOE_OK) return rc;
  return cuda_status(moe::launch_quantize_mx(src, batch, rows, cols, transpose != 0,
                                             static_cast<uint8_t *>(codes),
                                             static_cast<uint8_t *>(scales), true, stream));
}

int moe_quantize_weights(const moe_config *cfg, const void *w_bf16, int rows, int cols, int blocks_along_rows,
                         void *codes, void *scales, moe_stream_t stream) {
  Dims D;
  const int rc = check_config(cfg, &D);
  if (rc != MOE_OK) return rc;
  if (!D.mx) return MOE_ERR_ARG;
  return moe_quantize_mx(w_bf16, cfg->E, rows, cols, blocks_along_rows != 0, codes, scales, stream);
}

int moe_quantize_mx_both(const void *src, int batch, int rows, int cols, void *codes, void *scales,
                         void *codes_t, void *scales_t, moe_stream_t stream) {
  if (!src || !codes || !scales || !codes_t || !scales_t || batch <= 0 || rows <= 0 || cols <= 0)
    return MOE_ERR_ARG;
  if (rows % 128 || cols % 128) return MOE_ERR_SHAPE;
  if (!aligned16(src) || !aligned16(codes) || !aligned16(scales) || !aligned16(codes_t) ||
      !aligned16(scales_t))
    return MOE_ERR_ALIGN;
  DeviceInfo dev;
  const int rc = device_info(&dev);
  if (rc != MOE_OK) return rc;
  return cuda_status(moe::launch_quantize_mx_both(
      src, batch, rows, cols, static_cast<uint8_t *>(codes), static_cast<uint8_t *>(scales),
      static_cast<uint8_t *>(codes_t), static_cast<uint8_t *>(scales_t), true, stream));
}

int moe_prepare_weights(const moe_config *cfg, const void *w_gu, const void *w_dn, void *gu, void *gu_scale,
                        void *dn, void *dn_scale, void *gu_t, void *gu_t_scale, void *dn_t, void *dn_t_scale,
                        float *gu_gscale, float *dn_gscale, moe_stream_t stream) {
  Dims D;
  int rc = check_config(cfg, &D);
  if (rc != MOE_OK) return rc;
  if (!w_gu || !w_dn) return MOE_ERR_ARG;
  const bool bwd = gu_t != nullptr;
  if ((dn_t != nullptr) != bwd) return MOE_ERR_ARG;
  if (D.nv) {
    if (bwd || !gu || !gu_scale || !dn || !dn_scale || !gu_gscale || !dn_gscale) return MOE_ERR_ARG;
    const void *p[] = {w_gu, w_dn, gu, gu_scale, dn, dn_scale};
    for (const void *q : p)
      if (!aligned16(q)) return MOE_ERR_ALIGN;
    // one fp32 per expert: 4-byte alignment (an expert's slot of a per-layer array)
    if ((reinterpret_cast<uintptr_t>(gu_gscale) & 3u) || (reinterpret_cast<uintptr_t>(dn_gscale) & 3u))
      return MOE_ERR_ALIGN;
    DeviceInfo dev;
    if ((rc = device_info(&dev)) != MOE_OK) return rc;
    const long E = D.E, d = D.d, m = D.m;
    if ((rc = cuda_status(moe::launch_nv_global_scales(w_gu, D.E, 2 * m * d, gu_gscale, stream))) != MOE_OK ||
        (rc = cuda_status(moe::launch_nv_global_scales(w_dn, D.E, d * m, dn_gscale, stream))) != MOE_OK ||
        (rc = cuda_status(moe::launch_nv_quantize_rows(w_gu, E * 2 * m, D.d, 2 * m, gu_gscale,
                                                       static_cast<uint8_t *>(gu), static_cast<uint8_t *>(gu_scale),
                                                       true, stream))) != MOE_OK)
      return rc;
    return cuda_status(moe::launch_nv_quantize_rows(w_dn, E * d, D.m, d, dn_gscale, static_cast<uint8_t *>(dn),
                                                    static_cast<uint8_t *>(dn_scale), true, stream));
  }
  if (D.mx && (!gu || !gu_scale || !dn || !dn_scale || (bwd && (!gu_t_scale || !dn_t_scale)))) return MOE_ERR_ARG;
  const void *ptrs[] = {w_gu, w_dn, gu, gu_scale, dn, dn_scale, gu_t, gu_t_scale, dn_t, dn_t_scale};
  for (const void *q : ptrs)
    if (q && !aligned16(q)) return MOE_ERR_ALIGN;
  DeviceInfo dev;
  if ((rc = device_info(&dev)) != MOE_OK) return rc;
  const int E = D.E, d = D.d, m = D.m;
  auto u8 = [](void *p) { return static_cast<uint8_t *>(p); };
  if (D.mx) {
    if (bwd) {
      if ((rc = cuda_status(moe::launch_quantize_mx_both(w_gu, E, 2 * m, d, u8(gu), u8(gu_scale), u8(gu_t),
                                                         u8(gu_t_scale), false, stream))) != MOE_OK)
        return rc;
      return cuda_status(moe::launch_quantize_mx_both(w_dn, E, d, m, u8(dn), u8(dn_scale), u8(dn_t), u8(dn_t_scale),
                                                      false, stream));
    }
    if ((rc = cuda_status(moe::launch_quantize_mx(w_gu, E, 2 * m, d, false, u8(gu), u8(gu_scale), false, stream))) !=
        MOE_OK)
      return rc;
    return cuda_status(moe::launch_quantize_mx(w_dn, E, d, m, false, u8(dn), u8(dn_scale), false, stream));
  }
  // BF16 experts: the masters are the forward operands (copied when gu / dn name
  // other buffers); the backward reads per-expert transposes
  if (gu && gu != w_gu &&
      cudaMemcpyAsync(gu, w_gu, static_cast<size_t>(E) * 2 * m * d * 2, cudaMemcpyDeviceToDevice, stream) !=
          cudaSuccess)
    return MOE_ERR_CUDA;
  if (dn && dn != w_dn &&
      cudaMemcpyAsync(dn, w_dn, static_cast<size_t>(E) * d * m * 2, cudaMemcpyDeviceToDevice, stream) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (!bwd) return MOE_OK;
  if ((rc = cuda_status(moe::launch_transpose_bf16(w_gu, E, 2 * m, d, gu_t, stream))) != MOE_OK) return rc;
  return cuda_status(moe::launch_transpose_bf16(w_dn, E, d, m, dn_t, stream));
}

static int scales_layout(const void *src, int64_t rows, int32_t K, bool to_tiled, void *dst,
                         moe_stream_t stream) {
  if (!src || !dst || rows <= 0 || K <= 0) return MOE_ERR_ARG;
  if (src == dst) return MOE_ERR_ARG;
  if (rows % 128 || K % 128) return MOE_ERR_SHAPE;
  if (!aligned16(src) || !aligned16(dst)) return MOE_ERR_ALIGN;
  DeviceInfo dev;
  const int rc = device_info(&dev);
  if (rc != MOE_OK) return rc;
  return cuda_status(moe::launch_scales_layout(src, static_cast<long>(rows), K, to_tiled, dst, stream));
}

int moe_prepare_scales(const void *scales, int64_t rows, int32_t K, void *prepared, moe_stream_t stream) {
  return scales_layout(scales, rows, K, true, prepared, stream);
}

int moe_canonical_scales(const void *prepared, int64_t rows, int32_t K, void *scales, moe_stream_t stream) {
  return scales_layout(prepared, rows, K, false, scales, stream);
}

int moe_transpose_bf16(const void *src, int batch, int rows, int cols, void *dst,
                       moe_stream_t stream) {
  if (!src || !dst || batch <= 0 || rows <= 0 || cols <= 0) return MOE_ERR_ARG;
  if (rows % 32 || cols % 64) return MOE_ERR_SHAPE;
  if (!aligned16(src) || !aligned16(dst)) return MOE_ERR_ALIGN;
  DeviceInfo dev;
  const int rc = device_info(&dev);
  if (rc != MOE_OK) return rc;
  return cuda_status(moe::launch_transpose_bf16(src, batch, rows, cols, dst, stream));
}

static int route_impl(const Dims &D, const float *logits, const RouteBufs &rb, cudaStream_t s) {
  Traced tr("route_schedule", s);
  return cuda_status(moe::launch_route(logits, D.T, D.E, D.k, rb, s));
}

int moe_route(const moe_config *cfg, const float *logits, int32_t *idx, float *w, int32_t *counts,
              int32_t *offsets, int32_t *perm, void *ws, moe_stream_t stream) {
  Dims D;
  int rc = check_config(cfg, &D);
  if (rc != MOE_OK) return rc;
  if (!logits || !ws) return MOE_ERR_ARG;
  if (!aligned16(logits) || !aligned16(ws)) return MOE_ERR_ALIGN;
  DeviceInfo dev;
  if ((rc = device_info(&dev)) != MOE_OK) return rc;
  Layout W;
  ws_layout(D, W);
  Ptrs p = route_ptrs(D, W, ws, ws, W);
  if (idx) p.rb.idx = idx;
  if (w) p.rb.w = w;
  if (counts) p.rb.counts = counts;
  if (offsets) p.rb.offsets = offsets;
  if (perm) p.rb.perm = perm;
  if (cudaMemsetAsync(p.status, 0, 4, stream) != cudaSuccess) return MOE_ERR_CUDA;
  return route_impl(D, logits, p.rb, stream);
}

int moe_forward(const moe_config *cfg, const void *x, const float *logits, const moe_weights *Wt,
                void *y, void *saved, void *ws, moe_stream_t stream) {
  Dims D;
  int rc = check_config(cfg, &D);
  if (rc != MOE_OK) return rc;
  if (!x || !logits || !Wt || !y || !ws || !Wt->gu || !Wt->dn) return MOE_ERR_ARG;
  if ((D.mx || D.nv) && (!Wt->gu_scale || !Wt->dn_scale)) return MOE_ERR_ARG;
  if (D.nv && (!Wt->gu_gscale || !Wt->dn_gscale || saved)) return MOE_ERR_ARG;  // NVFP4: inference only
  if (D.ms && (!Wt->s_gu || !Wt->s_dn)) return MOE_ERR_ARG;
  if (!aligned16(x) || !aligned16(logits) || !aligned16(y) || !aligned16(ws) ||
      !aligned16(Wt->gu) || !aligned16(Wt->dn) || (saved && !aligned16(saved)) ||
      ((D.mx || D.nv) && (!aligned16(Wt->gu_scale) || !aligned16(Wt->dn_scale))) ||
      (D.ms && (!aligned16(Wt->s_gu) || !aligned16(Wt->s_dn))))
    return MOE_ERR_ALIGN;
  DeviceInfo dev;
  if ((rc = device_info(&dev)) != MOE_OK) return rc;
  cudaStream_t s = stream;
  Layout W, S;
  ws_layout(D, W);
  saved_layout(D, S);
  const bool train = saved != nullptr;
  const Layout &RL = train ? S : W;
  void *rbase = train ? saved : ws;
  Ptrs p = route_ptrs(D, RL, rbase, ws, W);
  const RouteBufs &rb = p.rb;
  if (cudaMemsetAsync(p.status, 0, 4, s) != cudaSuccess) return MOE_ERR_CUDA;

  // S1 + S2
  if ((rc = route_impl(D, logits, rb, s)) != MOE_OK) return rc;
  // load-balancing term (after the schedule: needs the counts)
  if (D.aux_alpha > 0.f) {
    Traced tr("balance_loss", s);
    float *grad = train ? reinterpret_cast<float *>(S.ptr(saved, "aux_grad")) : nullptr;
    rc = cuda_status(moe::launch_balance(logits, D.T, D.E, D.k, rb.counts, D.aux_alpha,
                                         reinterpret_cast<float *>(W.ptr(ws, "aux_part")), grad,
                                         reinterpret_cast<float *>(W.ptr(ws, "aux")), s));
    if (rc != MOE_OK) return rc;
  }
  // S3 dispatch gather (+ MX quantisation of x); with a ring it runs inside
  // the gate/up GEMM launch below.
  char *xs = D.ring ? W.ptr(ws, "ring") : W.ptr(ws, "xs");
  uint8_t *xs_sf = reinterpret_cast<uint8_t *>(D.ring ? W.ptr(ws, "ring_sf") : W.ptr(ws, "xs_sf"));
  uint8_t *xT = (train && D.mx) ? reinterpret_cast<uint8_t *>(S.ptr(saved, "xT")) : nullptr;
  uint8_t *xT_sf = (train && D.mx) ? reinterpret_cast<uint8_t *>(S.ptr(saved, "xT_sf")) : nullptr;
  uint8_t *xq = reinterpret_cast<uint8_t *>(W.ptr(ws, "xq"));
  uint8_t *xq_sf = reinterpret_cast<uint8_t *>(W.ptr(ws, "xq_sf"));
  if (D.nv) {
    // NVFP4: x's second-level scale, every token's codes once, then the rows
    Traced tr("dispatch_gather", s);
    float *xg = reinterpret_cast<float *>(W.ptr(ws, "x_gscale"));
    rc = cuda_status(moe::launch_nv_global_scales(x, 1, static_cast<long>(D.T) * D.d, xg, s));
    if (rc == MOE_OK)
      rc = cuda_status(moe::launch_nv_quantize_rows(x, D.T, D.d, D.T, xg, xq, xq_sf, false, s));
    if (rc == MOE_OK)
      rc = cuda_status(moe::launch_nv_gather(xq, xq_sf, D.d, D.k, D.E, rb, D.Rp, reinterpret_cast<uint8_t *>(xs),
                                             xs_sf, s));
  } else if (!D.ring) {
    Traced tr("dispatch_gather", s);
    rc = cuda_status(
        moe::launch_gather(x, D.T, D.d, D.k, D.E, rb, D.Rp, D.mx, xs, xs_sf, xT, xT_sf, xq, xq_sf, s));
  } else {
    // row-blocked codes once per token (identical for all k routed copies);
    // the ring kernel's gather SMs move them.  A training pass also needs the
    // column-blocked codes of the dispatched rows.
    {
      Traced tr("quantize_tokens", s);
      rc = cuda_status(moe::launch_quantize_tokens(x, D.T, D.d, xq, xq_sf, s));
    }
    if (rc == MOE_OK && train) {
      Traced tr("dispatch_xT", s);
      rc = cuda_status(
          moe::launch_gather(x, D.T, D.d, D.k, D.E, rb, D.Rp, true, nullptr, nullptr, xT, xT_sf, nullptr,
                             nullptr, s));
    }
  }
  if (rc != MOE_OK) return rc;
  // S4 gate/up GEMM + SwiGLU (+ MX quantisation of h)
  char *h_bf16 = (D.mx || D.nv) ? nullptr : (train ? S.ptr(saved, "h") : W.ptr(ws, "h"));
  char *GU = train ? S.ptr(saved, "GU") : nullptr;
  uint8_t *hq = reinterpret_cast<uint8_t *>(W.ptr(ws, "hq"));
  uint8_t *hq_sf = reinterpret_cast<uint8_t *>(W.ptr(ws, "hq_sf"));
  char *o = RL.ptr(rbase, "o");
  {
    Gemm q;
    q.mx = D.mx;
    q.bn = 256;
    q.epi = moe::EPI_SWIGLU;
    q.a = xs;
    q.a_rows = D.ring ? static_cast<long>(D.ring_slots) * 128 : D.Rp;
    q.b = Wt->gu;
    q.b_rows = static_cast<long>(D.E) * 2 * D.m;
    q.K = D.d;
    q.g = base_args(moe::SCHED_GROUP_M, D.E, rb.poff, p.status);
    q.g.K = D.d;
    q.g.n_tiles = D.m / 128;
    q.g.b_rows_per_group = 2 * D.m;
    q.g.b_split = D.m;
    q.g.sfa = xs_sf;
    q.g.sfa_kg = D.d / 128;
    q.g.sfb = static_cast<const uint8_t *>(Wt->gu_scale);
    q.g.sfb_kg = D.d / 128;
    q.g.out = h_bf16;
    q.g.ldo = D.m;
    q.g.out2 = GU;
    q.g.ldo2 = 2 * D.m;
    q.g.outq = (D.mx || D.nv) ? hq : nullptr;
    q.g.outq_sf = hq_sf;
    q.g.ldq = D.m;
    if (D.nv) {  // packed E2M1 operands: K-groups of the tiled scales are 64 wide
      q.mx = q.nv = true;
      q.g.sfa_kg = q.g.sfb_kg = D.d / 64;
      q.g.a_gscale = reinterpret_cast<const float *>(W.ptr(ws, "x_gscale"));
      q.g.b_gscale = Wt->gu_gscale;
    }
    if (train && D.mx) {
      q.g.outT = reinterpret_cast<uint8_t *>(S.ptr(saved, "hT"));
      q.g.outT_sf = reinterpret_cast<uint8_t *>(S.ptr(saved, "hT_sf"));
      q.g.ldT = D.Rp;
    }
    q.g.m_half = D.m;
    if (D.dump) {
      q.g.dump = reinterpret_cast<float *>(W.ptr(ws, "h_dump"));
      q.g.ld_dump = D.m;
    }
    if (D.starve) {
      q.g.debug_starve = 1;
      q.g.timeout_ns = kStarveTimeoutNs;
    }
    q.max_tiles = (D.Rp / 128) * q.g.n_tiles;
    q.out_rows = D.Rp;
    if (D.ring) {
      moe::RingArgs &r = q.g.ring;
      r.xq = xq;
      r.xq_sf = xq_sf;
      r.rb = rb;
      r.k = D.k;
      r.slots = D.ring_slots;
      r.codes = reinterpret_cast<uint8_t *>(xs);
      r.sf = xs_sf;
      int *ctrl = reinterpret_cast<int *>(W.ptr(ws, "ring_ctrl"));
      r.ready = ctrl;
      r.freed = ctrl + D.ring_slots;
      r.abort = ctrl + 2 * D.ring_slots;
      if (cudaMemsetAsync(ctrl, 0, (2 * static_cast<size_t>(D.ring_slots) + 1) * 4, s) != cudaSuccess)
        return MOE_ERR_CUDA;
      if ((rc = run_gemm_ring("dispatch_gemm1_ring", q, D, dev, s)) != MOE_OK) return rc;
    } else if ((rc = run_gemm("gemm1_gate_up_swiglu", q, dev, s)) != MOE_OK) {
      return rc;
    }
  }
  // S5 down GEMM
  {
    Gemm q;
    q.mx = D.mx;
    q.bn = bn_for(D.d);
    q.epi = moe::EPI_STORE;
    q.a = D.mx ? static_cast<const void *>(hq) : h_bf16;
    q.a_rows = D.Rp;
    q.b = Wt->dn;
    q.b_rows = static_cast<long>(D.E) * D.d;
    q.K = D.m;
    q.g = base_args(moe::SCHED_GROUP_M, D.E, rb.poff, p.status);
    q.g.K = D.m;
    q.g.n_tiles = D.d / q.bn;
    q.g.b_rows_per_group = D.d;
    q.g.sfa = hq_sf;
    q.g.sfa_kg = D.m / 128;
    q.g.sfb = static_cast<const uint8_t *>(Wt->dn_scale);
    q.g.sfb_kg = D.m / 128;
    q.g.out = o;
    q.g.ldo = D.d;
    if (D.nv) {  // h carries second-level scale 1 (a_gscale NULL)
      q.mx = q.nv = true;
      q.a = hq;
      q.g.sfa_kg = q.g.sfb_kg = D.m / 64;
      q.g.b_gscale = Wt->dn_gscale;
    }
    q.max_tiles = (D.Rp / 128) * q.g.n_tiles;
    q.out_rows = D.Rp;
    if ((rc = run_gemm("gemm2_down", q, dev, s)) != MOE_OK) return rc;
  }
  // S7 shared expert (BF16, dense over all tokens)
  char *s_out = nullptr;
  if (D.ms) {
    char *s_h = train ? S.ptr(saved, "s_h") : W.ptr(ws, "s_h");
    char *s_GU = train ? S.ptr(saved, "s_GU") : nullptr;
    s_out = W.ptr(ws, "s_out");
    Gemm q;
    q.mx = false;
    q.bn = 256;
    q.epi = moe::EPI_SWIGLU;
    q.a = x;
    q.a_rows = D.T;
    q.b = Wt->s_gu;
    q.b_rows = 2L * D.ms;
    q.K = D.d;
    q.g = base_args(moe::SCHED_DENSE, 1, nullptr, p.status);
    q.g.M = D.T;
    q.g.K = D.d;
    q.g.n_tiles = D.ms / 128;
    q.g.b_rows_per_group = 2 * D.ms;
    q.g.b_split = D.ms;
    q.g.out = s_h;
    q.g.ldo = D.ms;
    q.g.out2 = s_GU;
    q.g.ldo2 = 2 * D.ms;
    q.g.m_half = D.ms;
    q.max_tiles = (D.Tp / 128) * q.g.n_tiles;
    q.out_rows = D.Tp;
    if ((rc = run_gemm("shared_gemm1_gate_up_swiglu", q, dev, s)) != MOE_OK) return rc;
    Gemm q2;
    q2.mx = false;
    q2.bn = bn_for(D.d);
    q2.epi = moe::EPI_STORE;
    q2.a = s_h;
    q2.a_rows = D.Tp;
    q2.b = Wt->s_dn;
    q2.b_rows = D.d;
    q2.K = D.ms;
    q2.g = base_args(moe::SCHED_DENSE, 1, nullptr, p.status);
    q2.g.M = D.T;
    q2.g.K = D.ms;
    q2.g.n_tiles = D.d / q2.bn;
    q2.g.b_rows_per_group = D.d;
    q2.g.out = s_out;
    q2.g.ldo = D.d;
    q2.max_tiles = (D.Tp / 128) * q2.g.n_tiles;
    q2.out_rows = D.Tp;
    if ((rc = run_gemm("shared_gemm2_down", q2, dev, s)) != MOE_OK) return rc;
  }
  // S6 combine
  Traced tr("combine", s);
  return cuda_status(moe::launch_combine(o, s_out, D.T, D.d, D.k, D.E, rb, y, s));
}

int moe_backward(const moe_config *cfg, const void *dy, const void *x, const moe_weights *Wt,
                 const void *saved_c, void *dx, float *dlogits, void *dW_gu, void *dW_dn,
                 void *dWs_gu, void *dWs_dn, void *ws, moe_stream_t stream) {
  Dims D;
  int rc = check_config(cfg, &D);
  if (rc != MOE_OK) return rc;
  if (!D.bwd) return MOE_ERR_ARG;
  if (!dy || !x || !Wt || !saved_c || !dx || !dlogits || !dW_gu || !dW_dn || !ws) return MOE_ERR_ARG;
  if (!Wt->gu_t || !Wt->dn_t) return MOE_ERR_ARG;
  if (D.mx && (!Wt->gu_t_scale || !Wt->dn_t_scale)) return MOE_ERR_ARG;
  if (D.ms && (!Wt->s_gu_t || !Wt->s_dn_t || !dWs_gu || !dWs_dn)) return MOE_ERR_ARG;
  const void *ptrs[] = {dy, x, saved_c, dx, dlogits, dW_gu, dW_dn, ws, Wt->gu_t, Wt->dn_t};
  for (const void *q : ptrs)
    if (!aligned16(q)) return MOE_ERR_ALIGN;
  if (D.mx && (!aligned16(Wt->gu_t_scale) || !aligned16(Wt->dn_t_scale))) return MOE_ERR_ALIGN;
  if (D.ms && (!aligned16(Wt->s_gu_t) || !aligned16(Wt->s_dn_t) || !aligned16(dWs_gu) ||
               !aligned16(dWs_dn)))
    return MOE_ERR_ALIGN;
  DeviceInfo dev;
  if ((rc = device_info(&dev)) != MOE_OK) return rc;
  cudaStream_t s = stream;
  void *saved = const_cast<void *>(saved_c);
  Layout W, S;
  ws_layout(D, W);
  saved_layout(D, S);
  Ptrs p = route_ptrs(D, S, saved, ws, W);
  const RouteBufs &rb = p.rb;
  const int *nrows_dev = rb.poff + D.E;
  const bool mx = D.mx;
  auto u8 = [&](const char *n) { return reinterpret_cast<uint8_t *>(W.ptr(ws, n)); };

  char *o = S.ptr(saved, "o");
  char *GU = S.ptr(saved, "GU");
  char *h = S.ptr(saved, "h");
  float *g = reinterpret_cast<float *>(W.ptr(ws, "g"));
  char *dO = W.ptr(ws, "dO");
  char *dGU = W.ptr(ws, "dGU");
  char *dX = W.ptr(ws, "dX");

  // B1 reverse combine: dO = w * dy (bf16; MX row-quantised along d), g = <dy, o>
  {
    Traced tr("reverse_combine", s);
    if (mx)  // also writes dO^T's column-blocked codes (the wgrad operand)
      rc = cuda_status(moe::launch_reverse_combine_mx(dy, o, D.T, D.d, D.k, D.E, rb, D.Rp, g, u8("dOq"),
                                                      u8("dOq_sf"), u8("dOT"), u8("dOT_sf"), s));
    else
      rc = cuda_status(moe::launch_reverse_combine(dy, o, D.T, D.d, D.k, D.E, rb, D.Rp, dO, g, s));
  }
  if (rc != MOE_OK) return rc;
  // B2 dgrad of the down projection with the SwiGLU backward in the epilogue
  {
    Gemm q;
    q.mx = mx;
    // 256-column tiles (one TMEM accumulator; the epilogue reads it 64
    // columns at a time): measured faster than 128-column tiles with two
    // accumulators, which re-read the dO codes twice as often.
    q.bn = bn_for(D.m);
    q.epi = moe::EPI_SWIGLU_BWD;
    q.a = mx ? static_cast<const void *>(u8("dOq")) : dO;
    q.a_rows = D.Rp;
    q.b = Wt->dn_t;
    q.b_rows = static_cast<long>(D.E) * D.m;
    q.K = D.d;
    q.g = base_args(moe::SCHED_GROUP_M, D.E, rb.poff, p.status);
    q.g.K = D.d;
    q.g.n_tiles = D.m / q.bn;
    q.g.b_rows_per_group = D.m;
    q.g.sfa = u8("dOq_sf");
    q.g.sfa_kg = D.d / 128;
    q.g.sfb = static_cast<const uint8_t *>(Wt->dn_t_scale);
    q.g.sfb_kg = D.d / 128;
    // MXFP8: dGU only as codes, row-blocked (gate/up dgrad) and column-blocked
    // (gate/up wgrad), plus the bf16 values with the dump flag; BF16: dGU in bf16
    q.g.out = mx ? (D.dump ? W.ptr(ws, "dGU_dump") : nullptr) : dGU;
    q.g.ldo = 2 * D.m;
    q.g.outq = mx ? u8("dGUq") : nullptr;
    q.g.outq_sf = u8("dGUq_sf");
    q.g.ldq = 2 * D.m;
    if (mx) {
      q.g.outT = u8("dGUT");
      q.g.outT_sf = u8("dGUT_sf");
      q.g.ldT = D.Rp;
    }
    q.g.aux = GU;
    q.g.ld_aux = 2 * D.m;
    q.g.m_half = D.m;
    q.max_tiles = (D.Rp / 128) * q.g.n_tiles;
    q.out_rows = D.Rp;
    if ((rc = run_gemm("dgrad_down_swiglu_bwd", q, dev, s)) != MOE_OK) return rc;
  }
  // B4 dgrad of the gate/up projection
  {
    Gemm q;
    q.mx = mx;
    q.bn = bn_for(D.d);
    q.epi = moe::EPI_STORE;
    q.a = mx ? static_cast<const void *>(u8("dGUq")) : dGU;
    q.a_rows = D.Rp;
    q.b = Wt->gu_t;
    q.b_rows = static_cast<long>(D.E) * D.d;
    q.K = 2L * D.m;
    q.g = base_args(moe::SCHED_GROUP_M, D.E, rb.poff, p.status);
    q.g.K = 2 * D.m;
    q.g.n_tiles = D.d / q.bn;
    q.g.b_rows_per_group = D.d;
    q.g.sfa = u8("dGUq_sf");
    q.g.sfa_kg = 2 * D.m / 128;
    q.g.sfb = static_cast<const uint8_t *>(Wt->gu_t_scale);
    q.g.sfb_kg = 2 * D.m / 128;
    q.g.out = dX;
    q.g.ldo = D.d;
    q.max_tiles = (D.Rp / 128) * q.g.n_tiles;
    q.out_rows = D.Rp;
    if ((rc = run_gemm("dgrad_gate_up", q, dev, s)) != MOE_OK) return rc;
  }
  // Transposed bf16 wgrad operands of BF16 experts, K = padded rows.  With
  // MXFP8 experts their column-blocked codes were written by the kernels that
  // produced them: x^T by the dispatch, h^T by the gate/up GEMM, dO^T by B1,
  // dGU^T by B2.
  struct Tr {
    const void *src;
    int C;
    bool gather;
    const char *dst;
  } trs[] = {{dO, D.d, false, "dOT"}, {h, D.m, false, "hT"}, {dGU, 2 * D.m, false, "dGUT"}, {x, D.d, true, "xT"}};
  for (const Tr &t : trs) {
    if (mx) break;
    {
      Traced tr("transpose_wgrad_operands", s);
      rc = cuda_status(moe::launch_transpose_rows(t.src, t.C, 0, nrows_dev, D.Rp, t.gather, D.k, D.E,
                                                  &rb, D.Rp, W.ptr(ws, t.dst), D.Rp, s));
    }
    if (rc != MOE_OK) return rc;
  }
  // B3 wgrad of the down projection: dW_dn[e] = dO_e^T h_e
  {
    Gemm q;
    q.mx = mx;
    q.bn = bn_for(D.m);
    q.epi = moe::EPI_STORE;
    q.a = W.ptr(ws, "dOT");
    q.a_rows = D.d;
    q.b = mx ? S.ptr(saved, "hT") : W.ptr(ws, "hT");
    q.b_rows = D.m;
    q.K = D.Rp;
    q.g = base_args(moe::SCHED_GROUP_K, D.E, rb.poff, p.status);
    q.g.M = D.d;
    q.g.n_tiles = D.m / q.bn;
    q.g.sfa = u8("dOT_sf");
    q.g.sfa_kg = static_cast<int>(D.Rp / 128);
    q.g.sfb = mx ? reinterpret_cast<uint8_t *>(S.ptr(saved, "hT_sf")) : nullptr;
    q.g.sfb_kg = static_cast<int>(D.Rp / 128);
    q.g.out = dW_dn;
    q.g.ldo = D.m;
    q.max_tiles = static_cast<long>(D.E) * (D.d / 128) * q.g.n_tiles;
    q.out_rows = static_cast<long>(D.E) * (D.d);
    q.zero_dst = dW_dn;
    q.zero_expert_bytes = static_cast<long>(D.d) * D.m * 2;
    q.zero_counts = rb.counts;
    if ((rc = run_gemm("wgrad_down", q, dev, s)) != MOE_OK) return rc;
  }
  // B5 wgrad of the gate/up projection: dW_gu[e] = dGU_e^T X_e
  {
    Gemm q;
    q.mx = mx;
    q.bn = bn_for(D.d);
    q.epi = moe::EPI_STORE;
    q.a = W.ptr(ws, "dGUT");
    q.a_rows = 2L * D.m;
    q.b = mx ? S.ptr(saved, "xT") : W.ptr(ws, "xT");
    q.b_rows = D.d;
    q.K = D.Rp;
    q.g = base_args(moe::SCHED_GROUP_K, D.E, rb.poff, p.status);
    q.g.M = 2 * D.m;
    q.g.n_tiles = D.d / q.bn;
    q.g.sfa = u8("dGUT_sf");
    q.g.sfa_kg = static_cast<int>(D.Rp / 128);
    q.g.sfb = mx ? reinterpret_cast<uint8_t *>(S.ptr(saved, "xT_sf")) : u8("xT_sf");
    q.g.sfb_kg = static_cast<int>(D.Rp / 128);
    q.g.out = dW_gu;
    q.g.ldo = D.d;
    q.max_tiles = static_cast<long>(D.E) * (2 * D.m / 128) * q.g.n_tiles;
    q.out_rows = static_cast<long>(D.E) * (2 * D.m);
    q.zero_dst = dW_gu;
    q.zero_expert_bytes = 2L * D.m * D.d * 2;
    q.zero_counts = rb.counts;
    if ((rc = run_gemm("wgrad_gate_up", q, dev, s)) != MOE_OK) return rc;
  }
  // B7 shared expert backward (BF16, dense)
  char *s_dx = nullptr;
  if (D.ms) {
    char *s_GU = S.ptr(saved, "s_GU");
    char *s_h = S.ptr(saved, "s_h");
    char *s_dGU = W.ptr(ws, "s_dGU");
    s_dx = W.ptr(ws, "s_dx");
    {
      Gemm q;
      q.mx = false;
      q.bn = bn_for(D.ms);
      q.epi = moe::EPI_SWIGLU_BWD;
      q.a = dy;
      q.a_rows = D.T;
      q.b = Wt->s_dn_t;
      q.b_rows = D.ms;
      q.K = D.d;
      q.g = base_args(moe::SCHED_DENSE, 1, nullptr, p.status);
      q.g.M = D.T;
      q.g.K = D.d;
      q.g.n_tiles = D.ms / q.bn;
      q.g.b_rows_per_group = D.ms;
      q.g.out = s_dGU;
      q.g.ldo = 2 * D.ms;
      q.g.aux = s_GU;
      q.g.ld_aux = 2 * D.ms;
      q.g.m_half = D.ms;
      q.max_tiles = (D.Tp / 128) * q.g.n_tiles;
      q.out_rows = D.Tp;
      if ((rc = run_gemm("shared_dgrad_down_swiglu_bwd", q, dev, s)) != MOE_OK) return rc;
    }
    {
      Gemm q;
      q.mx = false;
      q.bn = bn_for(D.d);
      q.epi = moe::EPI_STORE;
      q.a = s_dGU;
      q.a_rows = D.Tp;
      q.b = Wt->s_gu_t;
      q.b_rows = D.d;
      q.K = 2L * D.ms;
      q.g = base_args(moe::SCHED_DENSE, 1, nullptr, p.status);
      q.g.M = D.T;
      q.g.K = 2 * D.ms;
      q.g.n_tiles = D.d / q.bn;
      q.g.b_rows_per_group = D.d;
      q.g.out = s_dx;
      q.g.ldo = D.d;
      q.max_tiles = (D.Tp / 128) * q.g.n_tiles;
      q.out_rows = D.Tp;
      if ((rc = run_gemm("shared_dgrad_gate_up", q, dev, s)) != MOE_OK) return rc;
    }
    struct TrS {
      const void *src;
      int C;
      long nsrc;
      const char *dst;
    } ts[] = {{dy, D.d, D.T, "s_dyT"},
              {s_h, D.ms, D.Tp, "s_hT"},
              {s_dGU, 2 * D.ms, D.Tp, "s_dGUT"},
              {x, D.d, D.T, "s_xT"}};
    for (const TrS &t : ts) {
      {
        Traced tr("shared_transpose_wgrad_operands", s);
        rc = cuda_status(moe::launch_transpose_rows(t.src, t.C, static_cast<int>(D.Tp), nullptr,
                                                    t.nsrc, false, D.k, D.E, nullptr, D.Tp,
                                                    W.ptr(ws, t.dst), D.Tp, s));
      }
      if (rc != MOE_OK) return rc;
    }
    {
      Gemm q;
      q.mx = false;
      q.bn = bn_for(D.ms);
      q.epi = moe::EPI_STORE;
      q.a = W.ptr(ws, "s_dyT");
      q.a_rows = D.d;
      q.b = W.ptr(ws, "s_hT");
      q.b_rows = D.ms;
      q.K = D.Tp;
      q.g = base_args(moe::SCHED_GROUP_K, 1, nullptr, p.status);
      q.g.M = D.d;
      q.g.K = static_cast<int>(D.Tp);
      q.g.n_tiles = D.ms / q.bn;
      q.g.out = dWs_dn;
      q.g.ldo = D.ms;
      q.max_tiles = (D.d / 128) * q.g.n_tiles;
      q.out_rows = static_cast<long>(1) * (D.d);
      if ((rc = run_gemm("shared_wgrad_down", q, dev, s)) != MOE_OK) return rc;
    }
    {
      Gemm q;
      q.mx = false;
      q.bn = bn_for(D.d);
      q.epi = moe::EPI_STORE;
      q.a = W.ptr(ws, "s_dGUT");
      q.a_rows = 2L * D.ms;
      q.b = W.ptr(ws, "s_xT");
      q.b_rows = D.d;
      q.K = D.Tp;
      q.g = base_args(moe::SCHED_GROUP_K, 1, nullptr, p.status);
      q.g.M = 2 * D.ms;
      q.g.K = static_cast<int>(D.Tp);
      q.g.n_tiles = D.d / q.bn;
      q.g.out = dWs_gu;
      q.g.ldo = D.d;
      q.max_tiles = (2L * D.ms / 128) * q.g.n_tiles;
      q.out_rows = static_cast<long>(1) * (2 * D.ms);
      if ((rc = run_gemm("shared_wgrad_gate_up", q, dev, s)) != MOE_OK) return rc;
    }
  }
  // B6 reverse dispatch + dlogits
  Traced tr("reverse_dispatch", s);
  const float *aux_grad = D.aux_alpha > 0.f ? reinterpret_cast<const float *>(S.ptr(saved, "aux_grad")) : nullptr;
  return cuda_status(
      moe::launch_reverse_dispatch(dX, s_dx, g, D.T, D.d, D.k, D.E, rb, dx, dlogits, aux_grad, s));
}

// ---------------------------------------------------------------- router projection
// The router GEMMs run on the library's own tcgen05 GEMM (DENSE schedule,
// single-CTA kernel).  Shapes the tiles do not cover (E not a multiple of the
// tile width, T not a multiple of 128) go through zero-padded copies in the
// workspace: Ep = E rounded up to 128, Tp = T rounded up to 128.
static long router_ep(const Dims &D) { return (D.E + 127L) / 128 * 128; }

int moe_router_forward(const moe_config *cfg, const void *x, const void *W_r, float *logits, void *ws,
                       moe_stream_t stream) {
  Dims D;
  int rc = check_config(cfg, &D);
  if (rc != MOE_OK) return rc;
  if (!x || !W_r || !logits || !ws) return MOE_ERR_ARG;
  if (!aligned16(x) || !aligned16(W_r) || !aligned16(logits) || !aligned16(ws)) return MOE_ERR_ALIGN;
  DeviceInfo dev;
  if ((rc = device_info(&dev)) != MOE_OK) return rc;
  Layout W;
  ws_layout(D, W);
  Traced tr("router_forward", stream);
  const long Ep = router_ep(D);
  float *lpad = reinterpret_cast<float *>(W.ptr(ws, "router_lpad"));  // [Tp, Ep]
  // logits [T, E] = x [T, d] W_r [E, d]^T, fp32 accumulation and output
  Gemm q;
  q.mx = false;
  q.bn = bn_for(Ep);
  q.epi = moe::EPI_STORE_F32;
  q.a = x;
  q.a_rows = D.T;
  q.b = W_r;
  q.b_rows = D.E;  // rows E .. Ep - 1 of the B tiles read as zero
  q.K = D.d;
  q.g = base_args(moe::SCHED_DENSE, 1, nullptr, reinterpret_cast<int *>(W.ptr(ws, "status")));
  q.g.M = D.T;
  q.g.K = D.d;
  q.g.n_tiles = static_cast<int>(Ep / q.bn);
  q.g.b_rows_per_group = static_cast<int>(Ep);
  q.g.out = lpad;
  q.g.ldo = Ep;
  q.max_tiles = (D.Tp / 128) * q.g.n_tiles;
  q.out_rows = D.Tp;
  if ((rc = run_gemm_single(q, dev, stream)) != MOE_OK) return rc;
  return cuda_status(moe::launch_crop_f32(lpad, D.T, D.E, Ep, logits, stream));
}

int moe_router_backward(const moe_config *cfg, const float *dlogits, const void *x, const void *W_r, void *dx,
                        void *dW_r, void *ws, moe_stream_t stream) {
  Dims D;
  int rc = check_config(cfg, &D);
  if (rc != MOE_OK) return rc;
  if (!dlogits || !x || !W_r || !dx || !dW_r || !ws) return MOE_ERR_ARG;
  if (!D.bwd) return MOE_ERR_ARG;
  if (!aligned16(dlogits) || !aligned16(x) || !aligned16(W_r) || !aligned16(dx) || !aligned16(dW_r) ||
      !aligned16(ws))
    return MOE_ERR_ALIGN;
  DeviceInfo dev;
  if ((rc = device_info(&dev)) != MOE_OK) return rc;
  Layout W;
  ws_layout(D, W);
  Traced tr("router_backward", stream);
  const long Ep = router_ep(D), Tp = D.Tp;
  int *status = reinterpret_cast<int *>(W.ptr(ws, "status"));
  char *G = W.ptr(ws, "router_g");      // [Tp, Ep] bf16(dlogits), zero-padded
  char *GT = W.ptr(ws, "router_gT");    // [Ep, Tp]
  char *WrT = W.ptr(ws, "router_WrT");  // [d, Ep] = W_r^T, zero-padded
  char *xT = W.ptr(ws, "router_xT");    // [d, Tp] = x^T, zero-padded
  if ((rc = cuda_status(moe::launch_pad_to_bf16(dlogits, D.T, D.E, static_cast<int>(Tp), static_cast<int>(Ep), G,
                                                stream))) != MOE_OK)
    return rc;
  if ((rc = cuda_status(moe::launch_transpose_rows(W_r, D.d, static_cast<int>(Ep), nullptr, D.E, false, D.k, D.E,
                                                   nullptr, Ep, WrT, Ep, stream))) != MOE_OK)
    return rc;
  // dx [T, d] = bf16(dx + g W_r): A = g [Tp, Ep], B = W_r^T [d, Ep], K = Ep
  {
    Gemm q;
    q.mx = false;
    q.bn = bn_for(D.d);
    q.epi = moe::EPI_ADD_BF16;
    q.a = G;
    q.a_rows = Tp;
    q.b = WrT;
    q.b_rows = D.d;
    q.K = Ep;
    q.g = base_args(moe::SCHED_DENSE, 1, nullptr, status);
    q.g.M = D.T;
    q.g.K = static_cast<int>(Ep);
    q.g.n_tiles = D.d / q.bn;
    q.g.b_rows_per_group = D.d;
    q.g.out = dx;
    q.g.ldo = D.d;
    q.g.aux = dx;
    q.g.ld_aux = D.d;
    q.max_tiles = (Tp / 128) * q.g.n_tiles;
    q.out_rows = D.T;
    if ((rc = run_gemm_single(q, dev, stream)) != MOE_OK) return rc;
  }
  // dW_r [E, d] = bf16(g^T x): A = g^T [Ep, Tp], B = x^T [d, Tp], K = Tp
  if ((rc = cuda_status(moe::launch_transpose_rows(G, static_cast<int>(Ep), static_cast<int>(Tp), nullptr, Tp,
                                                   false, D.k, D.E, nullptr, Tp, GT, Tp, stream))) != MOE_OK)
    return rc;
  if ((rc = cuda_status(moe::launch_transpose_rows(x, D.d, static_cast<int>(Tp), nullptr, D.T, false, D.k, D.E,
                                                   nullptr, Tp, xT, Tp, stream))) != MOE_OK)
    return rc;
  Gemm q;
  q.mx = false;
  q.bn = bn_for(D.d);
  q.epi = moe::EPI_STORE;
  q.a = GT;
  q.a_rows = Ep;
  q.b = xT;
  q.b_rows = D.d;
  q.K = Tp;
  q.g = base_args(moe::SCHED_DENSE, 1, nullptr, status);
  q.g.M = static_cast<int>(Ep);
  q.g.K = static_cast<int>(Tp);
  q.g.n_tiles = D.d / q.bn;
  q.g.b_rows_per_group = D.d;
  q.g.out = dW_r;
  q.g.ldo = D.d;
  q.max_tiles = (Ep / 128) * q.g.n_tiles;
  q.out_rows = D.E;
  return run_gemm_single(q, dev, stream);
}

int moe_get_status(void *ws, moe_stream_t stream) {
  if (!ws) return MOE_ERR_ARG;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return MOE_ERR_CUDA;
  int v = 0;
  if (cudaMemcpy(&v, ws, 4, cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaMemset(ws, 0, 4) != cudaSuccess) return MOE_ERR_CUDA;
  if (v & moe::kStatusTimeout) return MOE_ERR_TIMEOUT;
  return (v & moe::kStatusBounds) ? MOE_ERR_BOUNDS : MOE_OK;
}

int moe_trace_enable(int capacity) {
  if (capacity < 0) return MOE_ERR_ARG;
  trace_free();
  if (capacity == 0) return MOE_OK;
  g_trace.start = new cudaEvent_t[capacity];
  g_trace.end = new cudaEvent_t[capacity];
  g_trace.name = new const char *[capacity];
  for (int i = 0; i < capacity; ++i) {
    if (cudaEventCreate(&g_trace.start[i]) != cudaSuccess ||
        cudaEventCreate(&g_trace.end[i]) != cudaSuccess) {
      g_trace.capacity = i;
      trace_free();
      return MOE_ERR_CUDA;
    }
    g_trace.name[i] = nullptr;
  }
  g_trace.capacity = capacity;
  return MOE_OK;
}

void moe_trace_clear(void) { g_trace.count = 0; }

int moe_trace_count(void) { return g_trace.count; }

const char *moe_trace_name(int i) { return (i >= 0 && i < g_trace.count) ? g_trace.name[i] : nullptr; }

float moe_trace_ms(int i) {
  if (i < 0 || i >= g_trace.count) return -1.f;
  float ms = -1.f;
  if (cudaEventSynchronize(g_trace.end[i]) != cudaSuccess) return -1.f;
  if (cudaEventElapsedTime(&ms, g_trace.start[i], g_trace.end[i]) != cudaSuccess) return -1.f;
  return ms;
}

const char *moe_status_string(int status) {
  switch (status) {
    case MOE_OK: return "ok";
    case MOE_ERR_ARG: return "invalid argument";
    case MOE_ERR_SHAPE: return "unsupported shape";
    case MOE_ERR_ALIGN: return "pointer not 16-byte aligned";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_DEVICE: return "device is not sm_103";
    case MOE_ERR_TIMEOUT: return "a device-side wait timed out";
    case MOE_ERR_BOUNDS: return "a device-side bounds check failed (debug build)";
    default: return "unknown status";
  }
}

}  // extern "C"
