// mok_plan_noalloc: the schedule construction of mok_plan for caller-supplied routing,
// with its scratch in a fixed device array instead of the caller's workspace.
//
// Some callers cannot allocate device memory at all: code embedded in a host runtime that
// owns every device allocation, or code that must run where the allocator may not be
// called. They can still pass their inputs and outputs, but not a workspace. For them this
// entry point keeps the per-block expert histograms and slot ranks of the schedule builder
// in a file-scope __device__ array of kNoAllocScratchBytes, which every GPU that loads the
// library holds until the process exits.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "mok_internal.h"

namespace {

// 4 MiB: per-block histograms (ceil(T/32) * E int32) plus slot ranks (T*k int32).
constexpr size_t kNoAllocScratchBytes = size_t(4) << 20;

static __device__ __align__(256) int32_t g_plan_scratch[kNoAllocScratchBytes / sizeof(int32_t)];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
struct ScratchAddr {
  CUcontext ctx;   // the context the address belongs to
  void* ptr;
};
ScratchAddr g_scratch[kMaxDevices] = {};

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);

// cuCtxGetCurrent through the runtime's driver entry points (the library does not link
// the driver library itself).
CtxGetCurrentFn ctx_get_current_fn() {
  static CtxGetCurrentFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CtxGetCurrentFn>(p);
  });
  return fn;
}

// Device address of g_plan_scratch on the current device. In host code the symbol's name
// is only a host-side stand-in, so the address is looked up with the device current and
// cached per device, together with the context it was looked up in: a device reset (or any
// new primary context) loads the module again, possibly elsewhere, and the next call then
// finds another current context and looks the address up again.
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  CtxGetCurrentFn get = ctx_get_current_fn();
  if (!get) return cudaErrorDeviceUninitialized;
  CUcontext ctx = nullptr;
  if (get(&ctx) != CUDA_SUCCESS) return cudaErrorDeviceUninitialized;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!ctx || !g_scratch[dev].ptr || g_scratch[dev].ctx != ctx) {
    // the lookup also makes the device's primary context current when none is yet
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_plan_scratch);
    if (e != cudaSuccess) return e;
    if (get(&ctx) != CUDA_SUCCESS || !ctx) return cudaErrorDeviceUninitialized;
    g_scratch[dev] = ScratchAddr{ctx, p};
  }
  *out = g_scratch[dev].ptr;
  return cudaSuccess;
}

}  // namespace

extern "C" mok_status mok_plan_noalloc(mok_ctx_t ctx, mok_sched* sched, void* stream) {
  using namespace mok;
  const Dims* dp = ctx_dims(ctx);
  if (!dp) return MOK_ERR_INVALID_ARG;
  const Dims& d = *dp;
  if (d.router) return MOK_ERR_INVALID_ARG;  // routing must be supplied in sched
  if (!sched || !sched->topk_idx || !sched->gates || !sched->counts || !sched->offsets ||
      !sched->table || !sched->inv)
    return MOK_ERR_INVALID_ARG;
  if (!sched->aux || (reinterpret_cast<uintptr_t>(sched->aux) % 256) != 0)
    return MOK_ERR_WORKSPACE;
  const size_t hist_bytes = sizeof(int32_t) * (size_t)d.nblk * d.E;
  const size_t hist_room = align_up(hist_bytes, 256);
  const size_t need = hist_room + sizeof(int32_t) * (size_t)d.R;
  if (need > kNoAllocScratchBytes) return MOK_ERR_UNSUPPORTED;  // beyond the fixed scratch
  if (ctx_num_sms(ctx) <= 0) return MOK_ERR_CUDA;
  void* base = nullptr;
  if (scratch_address(&base) != cudaSuccess) return MOK_ERR_CUDA;
  int32_t* hist = static_cast<int32_t*>(base);
  int32_t* lrank = reinterpret_cast<int32_t*>(static_cast<char*>(base) + hist_room);
  // Both regions are fully rewritten before they are read (every block writes all E of
  // its histogram entries, every slot its rank), so nothing needs clearing between calls.
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  AuxPtrs a = aux_ptrs(d, sched->aux);
  if (cudaMemsetAsync(a.status, 0, sizeof(uint32_t), s) != cudaSuccess) return MOK_ERR_CUDA;
  if (launch_topk_rank(d, nullptr, sched->topk_idx, sched->gates, hist, lrank, a.status, s) !=
      cudaSuccess)
    return MOK_ERR_CUDA;
  if (launch_plan_scan(d, hist, sched->counts, sched->offsets, a, s) != cudaSuccess)
    return MOK_ERR_CUDA;
  if (launch_plan_macro(d, hist, sched->counts, sched->offsets, a, s) != cudaSuccess)
    return MOK_ERR_CUDA;
  if (launch_plan_scatter(d, sched->topk_idx, hist, lrank, sched->offsets, sched->table,
                          sched->inv, s) != cudaSuccess)
    return MOK_ERR_CUDA;
  return MOK_OK;
}
