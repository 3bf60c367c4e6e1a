// lmhead_compact_noalloc: the stable compaction of lmhead_compact for callers
// that cannot hand the library a workspace.
//
// Some callers have no way to obtain device memory of their own: a plugin or
// hook that runs inside a host framework whose caching allocator owns all of
// the GPU's memory, or a long-running service that reserves its memory at
// start-up and must not allocate afterwards (cudaMalloc may synchronise the
// device and can fail with out-of-memory in the middle of a run).  For them
// this entry point keeps its scratch -- the per-block counts of kept rows --
// in a fixed array that is part of the library image on every GPU that loads
// it, so the caller passes only its inputs and outputs.
//
// The scratch is shared by every call on a device and keeps the last call's
// contents.  Each call writes every count it later reads before reading it,
// so nothing has to start at zero; the one value that must (the device status
// word) is a caller output and is cleared by each call.  Two calls whose work
// overlaps on the GPU (different streams, or different host threads on one
// stream without ordering) race on the shared array: order them.
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/lmhead.h"
#include "internal.h"

namespace lmhead {
namespace {

constexpr int kNoallocRowsPerBlock = kCompactRowsPerBlock;  // rows per scan block
constexpr int kNoallocMaxBlocks =
    static_cast<int>(LMHEAD_NOALLOC_MAX_ROWS / kNoallocRowsPerBlock);  // 4096 counts = 16 KiB

static_assert(LMHEAD_NOALLOC_MAX_ROWS % kNoallocRowsPerBlock == 0,
              "maximum rows must be a whole number of scan blocks");

// Per-block kept-row counts of the compaction scan (the only scratch).
static __device__ __align__(256) int32_t g_noalloc_counts[kNoallocMaxBlocks];

// Device address of g_noalloc_counts, looked up once per device and CUDA
// context.  The address belongs to the module loaded in one context: a
// caller that makes another context current on the device, or a
// cudaDeviceReset that destroys the primary context and loads the module
// again, gets a fresh look-up.  Contexts are told apart by their unique id
// (cuCtxGetId), which is never reused within a process, so a new context
// never matches a stale entry even if its handle value repeats.
struct ScratchAddr {
  unsigned long long ctx_id = 0;
  int32_t* ptr = nullptr;
  bool ready = false;
};
constexpr int kMaxDevices = 64;
ScratchAddr g_scratch[kMaxDevices];
std::mutex g_scratch_mu;

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

// Unique id of the current CUDA context (driver entry points reached through
// the runtime, so the library needs no libcuda link).
bool current_context_id(unsigned long long* id) {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CtxGetCurrentFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(p);
  });
  CUcontext ctx = nullptr;
  if (get_current == nullptr || get_id == nullptr || get_current(&ctx) != CUDA_SUCCESS ||
      ctx == nullptr)
    return false;
  return get_id(ctx, id) == CUDA_SUCCESS;
}

lmhead_status scratch_for_current_device(int32_t** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return LMHEAD_ECUDA;
  std::lock_guard<std::mutex> g(g_scratch_mu);
  ScratchAddr& e = g_scratch[dev];
  unsigned long long ctx = 0;
  if (e.ready && current_context_id(&ctx) && ctx == e.ctx_id) {
    *out = e.ptr;
    return LMHEAD_OK;
  }
  // Set-up for this device and context.  In host code g_noalloc_counts names
  // a host-side shadow, not device memory; the device address must come from
  // the runtime (which also makes the device's context current if no context
  // was yet).
  e.ready = false;
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_noalloc_counts) != cudaSuccess || p == nullptr) {
    cudaGetLastError();  // leave no error behind for the next runtime call
    return LMHEAD_ECUDA;
  }
  if (!current_context_id(&ctx)) return LMHEAD_ECUDA;
  e.ptr = static_cast<int32_t*>(p);
  e.ctx_id = ctx;
  e.ready = true;
  *out = e.ptr;
  return LMHEAD_OK;
}

}  // namespace
}  // namespace lmhead

extern "C" lmhead_status lmhead_compact_noalloc(const uint8_t* keep, const int64_t* targets,
                                                int64_t N, int V, int32_t* idx,
                                                int32_t* targets_c, int32_t* d_nk,
                                                int32_t* d_status, lmhead_stream_t stream) {
  using namespace lmhead;
  if (N < 0 || V < 1 || targets == nullptr || idx == nullptr || targets_c == nullptr ||
      d_nk == nullptr || d_status == nullptr)
    return LMHEAD_EINVAL;
  if (N > LMHEAD_NOALLOC_MAX_ROWS) return LMHEAD_EINVAL;
  int major = 0, minor = 0, dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
      major != 10 || minor != 3)
    return LMHEAD_EUNSUPPORTED;
  if (!device_ptrs_ok({keep, targets, idx, targets_c, d_nk, d_status})) return LMHEAD_EINVAL;
  int32_t* counts = nullptr;
  lmhead_status st = scratch_for_current_device(&counts);
  if (st != LMHEAD_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(d_status, 0, sizeof(int32_t), s) != cudaSuccess) return LMHEAD_ECUDA;
  if (N == 0) {
    return cudaMemsetAsync(d_nk, 0, sizeof(int32_t), s) == cudaSuccess ? LMHEAD_OK
                                                                        : LMHEAD_ECUDA;
  }
  if (launch_compact(keep, targets, N, V, 0, idx, targets_c, d_nk, counts, d_status, s) !=
      cudaSuccess)
    return LMHEAD_ECUDA;
  return LMHEAD_OK;
}
