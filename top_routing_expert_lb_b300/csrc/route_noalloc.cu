// moe_route_noalloc: the router for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc or hand over a workspace: code that runs
// inside a host framework owning every byte of device memory through its own
// pool, plug-ins loaded into such a process, or code paths where allocating
// (and the device synchronisation it may imply) is not allowed.  For them this
// entry point runs the same router kernel as moe_route (logits, Top-k and the
// reduction of the side outputs in one launch), with the scratch it needs
// (the status word, per-expert accumulators, per-tile lse^2 sums and the
// finished-tile counter) placed in one file-scope device array instead of a
// caller workspace.  It never splits a tile's d dimension across CTAs (that
// would need partial logits of up to tens of MB), so shapes with few tokens
// use fewer SMs than through moe_route.
//
// That array is part of the library image: every GPU that loads the library
// holds it until the process exits.  All calls share it and it keeps the
// contents of the last call, so each call clears the words that must start at
// zero (and the router leaves its accumulators at zero); two calls that
// overlap on the GPU (different streams, no ordering)
// race on it.  The first call on a device looks up the array's device address
// (cudaGetSymbolAddress, with that device current) and caches it; make that
// first call before any stream capture.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/moe.h"
#include "moe_internal.h"

namespace moe {
namespace {

constexpr int kNoAllocMaxTokens = MOE_NOALLOC_MAX_TOKENS;
constexpr int kNoAllocMaxTiles = kNoAllocMaxTokens / kTileTokens;
constexpr int kNoAllocMaxExperts = MOE_MAX_EXPERTS;

// Byte offsets inside the static scratch (about 8 KB).
constexpr size_t kOffStatus = 0;   // int status word
constexpr size_t kOffAcc = 256;    // router accumulators: counts [256] int32 at +0, P sums
                                   // [256] u64 at +1024, entropy u64 at +5120, finished
                                   // tiles int32 at +5128 (5376 bytes)
constexpr size_t kAccBytes = 5376;
constexpr size_t kOffLse2 = kOffAcc + kAccBytes;  // [tiles] sums of lse^2
constexpr size_t kScratchBytes = kOffLse2 + static_cast<size_t>(kNoAllocMaxTiles) * 4;
static_assert(kNoAllocMaxExperts <= 256, "accumulator block holds 256 experts");

static __device__ __align__(256) unsigned char g_route_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
// Device address of the array and SM count, per device.  The address is
// published (release) after the SM count is stored, so a reader that sees it
// also sees the count; the set-up itself runs under a mutex, once per device.
std::atomic<unsigned char*> g_scratch_dev[kMaxDevices];
std::atomic<int> g_sm_count[kMaxDevices];
std::mutex g_setup_mutex;

// Per-device set-up: the device address of the static array (host code may
// not use the symbol itself as a device pointer) and the SM count.
int scratch_for_current_device(unsigned char** ptr, int* num_sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return MOE_ERR_CUDA;
  unsigned char* base = g_scratch_dev[dev].load(std::memory_order_acquire);
  if (base == nullptr) {
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    base = g_scratch_dev[dev].load(std::memory_order_acquire);
    if (base == nullptr) {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_route_scratch) != cudaSuccess || p == nullptr)
        return MOE_ERR_CUDA;
      int n = 0;
      if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
          n <= 0)
        return MOE_ERR_CUDA;
      g_sm_count[dev].store(n, std::memory_order_relaxed);
      base = static_cast<unsigned char*>(p);
      g_scratch_dev[dev].store(base, std::memory_order_release);
    }
  }
  *ptr = base;
  *num_sms = g_sm_count[dev].load(std::memory_order_relaxed);
  return MOE_OK;
}

inline bool aligned16(const void* q) { return (reinterpret_cast<uintptr_t>(q) & 15u) == 0; }

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" int moe_route_noalloc(const moe_shape_t* s, const uint16_t* x,
                                 const uint16_t* w_router, const float* logit_offset,
                                 const float* sel_bias, int32_t* ids, float* gates,
                                 int32_t* counts, float* f, float* P, float* bal_loss,
                                 float* z_loss, void* stream) {
  size_t unused = 0;
  int rc = moe_workspace_size(s, &unused);  // shape checks only
  if (rc != MOE_OK) return rc;
  if (s->flags & MOE_FLAG_EXPERT_CHOICE) return MOE_ERR_INVALID_ARG;
  if (s->T > kNoAllocMaxTokens || s->E > kNoAllocMaxExperts) return MOE_ERR_UNSUPPORTED;
  if (!counts || !f || !P || !bal_loss || !z_loss) return MOE_ERR_INVALID_ARG;
  if (s->T > 0) {
    if (!x || !w_router || !aligned16(x) || !aligned16(w_router)) return MOE_ERR_INVALID_ARG;
    if (s->k > 0 && (!ids || !gates)) return MOE_ERR_INVALID_ARG;
  }
  unsigned char* scratch = nullptr;
  int num_sms = 0;
  if ((rc = scratch_for_current_device(&scratch, &num_sms)) != MOE_OK) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // the status word and the accumulators start at zero on every call (the
  // router also leaves them at zero, unless a bounded wait ran out)
  if (cudaMemsetAsync(scratch, 0, kOffLse2, st) != cudaSuccess) return MOE_ERR_CUDA;
  uint8_t* acc = scratch + kOffAcc;
  RouterArgs ra{};
  ra.T = s->T;
  ra.d = s->d;
  ra.E = s->E;
  ra.k = s->k;
  ra.logit_offset = logit_offset;
  ra.sel_bias = sel_bias;
  ra.ids = ids;
  ra.gates = gates;
  ra.status = reinterpret_cast<int*>(scratch + kOffStatus);
  // the same wait limit as the workspace entry points, and only the router's
  // own variant bits (capacity and expert-choice bits do not concern it)
  ra.timeout_ns = s->tuning.wait_timeout_ns != 0 ? s->tuning.wait_timeout_ns
                                                  : default_wait_timeout_ns();
  ra.flags = s->flags & (kRouteSigmoid | kRouteNoRenorm);
  ra.max_split = 1;
  ra.acc_count = reinterpret_cast<int*>(acc);
  ra.acc_psum = reinterpret_cast<unsigned long long*>(acc + 1024);
  ra.tiles_done = reinterpret_cast<int*>(acc + 5128);
  ra.tile_lse2 = reinterpret_cast<float*>(scratch + kOffLse2);
  ra.C = -1;
  ra.balance_coef = s->balance_coef;
  ra.counts = counts;
  ra.f = f;
  ra.P = P;
  ra.bal_loss = bal_loss;
  ra.z_loss = z_loss;
  CUtensorMap mx, mw;
  std::memset(&mx, 0, sizeof(mx));
  std::memset(&mw, 0, sizeof(mw));
  if (s->T > 0) {
    const uint32_t nr = static_cast<uint32_t>((s->E + 15) / 16 * 16);
    if (!make_tmap_bf16(&mx, x, s->T, s->d, 128)) return MOE_ERR_CUDA;
    if (!make_tmap_bf16(&mw, w_router, s->E, s->d, nr)) return MOE_ERR_CUDA;
  }
  rc = launch_router(mx, mw, ra, num_sms, st);
  if (rc != 0) return rc == -2 ? MOE_ERR_UNSUPPORTED : MOE_ERR_CUDA;
  return MOE_OK;
}
