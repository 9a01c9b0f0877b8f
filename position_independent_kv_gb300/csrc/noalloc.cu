// rk_seg_attn_forward_noalloc: the forward for callers that must not
// allocate device memory when they call it.
//
// Who needs this: serving engines that reserve all device memory up front
// and forbid allocations on the request path, and code whose allocator is
// not reachable from where the forward is issued.  rk_seg_attn_forward asks
// such callers for a workspace (the split-over-segments kernel's partial
// outputs, partial LSEs and tickets); this entry point instead keeps that
// scratch in one file-scope device array of RK_NOALLOC_SCRATCH_BYTES, so the
// call itself allocates nothing.
//
// Costs and rules:
//  * the array exists on every GPU that loads this library's module and is
//    held until the process exits;
//  * every call on a device shares the one array and it keeps the previous
//    call's contents; the tickets that must start at zero are cleared by
//    each call (an asynchronous memset on the caller's stream);
//  * calls whose kernels overlap on the GPU (different streams without an
//    ordering between them) race on the array: order them;
//  * the first call on a device looks up the array's device address
//    (cudaGetSymbolAddress) with that device current and caches it with the
//    id of the device's current context; a later call that finds another
//    context there (after cudaDeviceReset the module is loaded again and the
//    array has a new address) looks it up again.  Make the first call on a
//    device, and the first call after a reset, before any stream capture;
//  * a plan whose scratch needs more than the array holds is refused with
//    RK_ERR_CAPACITY before anything is launched.
// The kernels and their arguments are exactly those of rk_seg_attn_forward.

#include <cudaTypedefs.h>

#include <mutex>

#include "rk_internal.h"

namespace {

constexpr size_t kScratchBytes = RK_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 128;

static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

std::mutex g_mu;
void* g_addr[kMaxDevices] = {};
unsigned long long g_ctx[kMaxDevices] = {};

// Id of the calling thread's current context (driver entry points, so the
// library keeps no link-time dependency on libcuda).
bool current_context_id(unsigned long long* id) {
  static PFN_cuCtxGetCurrent_v4000 get_cur = nullptr;
  static PFN_cuCtxGetId_v12000 get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 4000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_cur = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(f);
    f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(f);
  });
  CUcontext ctx = nullptr;
  if (!get_cur || !get_id || get_cur(&ctx) != CUDA_SUCCESS || !ctx) return false;
  return get_id(ctx, id) == CUDA_SUCCESS;
}

// Device address of g_scratch on the current device `dev`, looked up once
// per device and context.
rk_status_t scratch_address(int dev, void** out) {
  if (dev < 0 || dev >= kMaxDevices) return RK_ERR_CAPACITY;
  unsigned long long ctx = 0;
  if (!current_context_id(&ctx)) return RK_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_addr[dev] || g_ctx[dev] != ctx) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || !p) return RK_ERR_CUDA;
    g_addr[dev] = p;
    g_ctx[dev] = ctx;
  }
  *out = g_addr[dev];
  return RK_OK;
}

}  // namespace

extern "C" rk_status_t rk_seg_attn_forward_noalloc(rk_seg_attn_plan_t p, const void* q,
                                                   void* out, float* lse, void* stream) {
  if (!p || !q || !out || !lse) return RK_ERR_NULL;
  if (p->host_only) return RK_ERR_PLAN_MISMATCH;
  auto mis = [](const void* x) { return (reinterpret_cast<uintptr_t>(x) & 15) != 0; };
  if (mis(q) || mis(out) || (reinterpret_cast<uintptr_t>(lse) & 3)) return RK_ERR_ALIGNMENT;
  if (p->workspace_bytes > kScratchBytes) return RK_ERR_CAPACITY;
  int cur = -1;
  if (cudaGetDevice(&cur) != cudaSuccess) return RK_ERR_CUDA;
  if (cur != p->device) return RK_ERR_PLAN_MISMATCH;
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  rk::KernelArgs a{};
  rk::fill_args(*p, a, q, out, lse);
  if (p->num_parts) {
    void* base = nullptr;
    rk_status_t st = scratch_address(cur, &base);
    if (st != RK_OK) return st;
    st = rk::bind_workspace(*p, a, base, s);  // the layout rk_seg_attn_forward uses
    if (st != RK_OK) return st;
  }
  return rk::launch_forward(*p, a, q, s) == cudaSuccess ? RK_OK : RK_ERR_CUDA;
}
