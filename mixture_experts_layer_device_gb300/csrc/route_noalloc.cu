// moe_route_noalloc: the router top-k + schedule of moe_route for callers that
// cannot allocate device memory, e.g. code running inside a host framework that
// owns every device byte through its own arena, or a latency-critical path on
// which cudaMalloc (which can synchronise the device) is not acceptable.  Its
// scratch lives in a fixed-size array in this module's device memory, which
// every GPU that loads the library holds until the process exits.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/moe.h"
#include "kernels.h"

namespace {

constexpr long kMaxSlots = MOE_ROUTE_NOALLOC_MAX_SLOTS;     // T * k
constexpr int kMaxExperts = MOE_ROUTE_NOALLOC_MAX_EXPERTS;
constexpr long kMaxChunks = (kMaxSlots + moe::kSchedChunk - 1) / moe::kSchedChunk;
constexpr size_t kHistBytes = static_cast<size_t>(kMaxChunks) * kMaxExperts * sizeof(int);
constexpr size_t kInvBytes = static_cast<size_t>(kMaxSlots) * sizeof(int);
constexpr size_t kPoffBytes = ((kMaxExperts + 1) * sizeof(int) + 255) / 256 * 256;
constexpr size_t kScratchBytes = kHistBytes + kInvBytes + kPoffBytes;

// Per-chunk expert histograms, the row -> slot inverse permutation and the
// padded offsets of the schedule.  Every byte a call reads is written earlier
// in the same call, so nothing has to start at zero.
static __device__ __align__(256) unsigned char g_route_scratch[kScratchBytes];

std::mutex g_mu;
void *g_scratch_dev[64] = {};

// Device address of the scratch array on the current device, looked up once per
// device (the first call on a device does this set-up) and kept for the life of
// the process; it is not looked up again after a device reset.
int scratch_address(void **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MOE_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_dev[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_route_scratch) != cudaSuccess || !p) return MOE_ERR_CUDA;
    g_scratch_dev[dev] = p;
  }
  *out = g_scratch_dev[dev];
  return MOE_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" int moe_route_noalloc(const moe_config *cfg, const float *logits, int32_t *idx, float *w,
                                 int32_t *counts, int32_t *offsets, int32_t *perm,
                                 moe_stream_t stream) {
  if (!cfg || !logits || !idx || !w || !counts || !offsets || !perm) return MOE_ERR_ARG;
  if (cfg->T <= 0 || cfg->E <= 0 || cfg->k <= 0) return MOE_ERR_ARG;
  if (cfg->k > cfg->E || cfg->k > 16) return MOE_ERR_SHAPE;
  if (cfg->E > kMaxExperts || static_cast<long>(cfg->T) * cfg->k > kMaxSlots) return MOE_ERR_SHAPE;
  if (!aligned16(logits) || !aligned16(idx) || !aligned16(w) || !aligned16(counts) ||
      !aligned16(offsets) || !aligned16(perm))
    return MOE_ERR_ALIGN;
  int major = 0, minor = 0, dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (major != 10 || minor != 3) return MOE_ERR_DEVICE;
  void *base = nullptr;
  const int rc = scratch_address(&base);
  if (rc != MOE_OK) return rc;
  char *b = static_cast<char *>(base);
  moe::RouteBufs rb = {};
  rb.idx = idx;
  rb.w = w;
  rb.counts = counts;
  rb.offsets = offsets;
  rb.perm = perm;
  rb.hist = reinterpret_cast<int *>(b);
  rb.inv = reinterpret_cast<int *>(b + kHistBytes);
  rb.poff = reinterpret_cast<int *>(b + kHistBytes + kInvBytes);
  rb.n_tok = cfg->T;
  rb.n_slots = static_cast<long>(cfg->T) * cfg->k;
  return moe::launch_route(logits, cfg->T, cfg->E, cfg->k, rb, stream) == cudaSuccess ? MOE_OK
                                                                                     : MOE_ERR_CUDA;
}
