// Init-routing for callers that cannot allocate device memory.
//
// Some callers of this library run where cudaMalloc is off limits: code that
// executes inside a memory pool or allocator callback, a runtime whose device
// memory is fully pre-reserved and handed out by someone else, or a host
// thread that must not take the allocator's locks on its latency-critical
// path.  moe_init_routing asks the caller for a workspace; this variant needs
// none.  Its scratch (the per-chunk expert histograms and their starting
// positions) lives in the file-scope device array below, which every GPU that
// loads the library keeps for the life of the process.
//
// Limits and sharing rules (also stated in include/moe.h):
//  - the array holds kStaticScratchBytes (1 MiB): 2 * n_chunks * E int32
//    values, where n_chunks = ceil(T*k / CH) <= 256 is set by the same chunking
//    as moe_init_routing; larger problems are rejected with
//    MOE_ERR_UNSUPPORTED before anything is launched;
//  - every call on a device uses the same array and leaves its contents in
//    place.  Nothing in it needs to start at zero (each call writes every
//    value it later reads), but two calls whose kernels overlap on the GPU --
//    on different streams, or from different host threads -- race on it;
//  - the first call on a device looks up the array's device address
//    (cudaGetSymbolAddress) with that device current and caches it; make that
//    first call before any stream capture begins.
#include <atomic>
#include <mutex>

#include "moe_common.cuh"
#include "moe_internal.h"

namespace {

constexpr size_t kStaticScratchBytes = size_t(1) << 20;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) int32_t g_routing_scratch[kStaticScratchBytes / sizeof(int32_t)];

// Per device, the array's device address once it has been looked up.  Reads take no lock; the
// mutex is taken only by a call that finds no address yet for its device.
std::atomic<int32_t*> g_scratch_ptr[kMaxDevices] = {};
std::mutex g_mutex;

// Device address of g_routing_scratch on the current device (looked up once per device).
int scratch_for_current_device(int32_t** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return MOE_ERR_UNSUPPORTED;
  int32_t* p = g_scratch_ptr[dev].load(std::memory_order_acquire);
  if (p == nullptr) {
    std::lock_guard<std::mutex> lock(g_mutex);
    p = g_scratch_ptr[dev].load(std::memory_order_relaxed);
    if (p == nullptr) {
      void* a = nullptr;
      if (cudaGetSymbolAddress(&a, g_routing_scratch) != cudaSuccess || a == nullptr) return MOE_ERR_CUDA;
      p = static_cast<int32_t*>(a);
      g_scratch_ptr[dev].store(p, std::memory_order_release);
    }
  }
  *out = p;
  return MOE_OK;
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" int moe_init_routing_static_scratch(const int32_t* topk_idx, int T, int E, int k, const uint16_t* x,
                                               int H, uint16_t* x_exp, int32_t* counts, int32_t* offsets,
                                               int32_t* sorted_pair, int32_t* pair_pos, void* stream) {
  if (T < 0 || E < 1 || k < 1) return MOE_ERR_INVALID_ARG;
  if (E > 1024 || k > 32 || k > E || (long long)T * k >= (1LL << 31)) return MOE_ERR_UNSUPPORTED;
  if (!counts || !offsets) return MOE_ERR_INVALID_ARG;
  if ((x == nullptr) != (x_exp == nullptr)) return MOE_ERR_INVALID_ARG;
  if (x) {
    if (H <= 0) return MOE_ERR_INVALID_ARG;
    if (H % 64 != 0) return MOE_ERR_UNSUPPORTED;
    if (!aligned16(x) || !aligned16(x_exp)) return MOE_ERR_INVALID_ARG;
  }
  if (!aligned16(counts) || !aligned16(offsets)) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!topk_idx || !sorted_pair || !pair_pos || !aligned16(topk_idx) || !aligned16(sorted_pair) ||
                !aligned16(pair_pos)))
    return MOE_ERR_INVALID_ARG;
  const int P = T * k;
  if (moe::routing_scratch_bytes(P, E) > kStaticScratchBytes) return MOE_ERR_UNSUPPORTED;
  int32_t* scratch = nullptr;
  const int s = scratch_for_current_device(&scratch);
  if (s != MOE_OK) return s;
  const cudaError_t e = moe::launch_init_routing(topk_idx, P, E, k, x, H, x_exp, counts, offsets, sorted_pair,
                                                 pair_pos, scratch, nullptr, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
