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
//    (cudaGetSymbolAddress) with that device current and caches it; make
//    that first call before any stream capture;
//  * a plan whose scratch needs more than the array holds is refused with
//    RK_ERR_CAPACITY before anything is launched.
// The kernels and their arguments are exactly those of rk_seg_attn_forward.

#include <mutex>

#include "rk_internal.h"

namespace {

constexpr size_t kScratchBytes = RK_NOALLOC_SCRATCH_BYTES;
constexpr int kSplitHeads = 8;
constexpr int kMaxDevices = 128;

static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

std::mutex g_mu;
void* g_addr[kMaxDevices] = {};

// Device address of g_scratch on the current device `dev` (cached).
rk_status_t scratch_address(int dev, void** out) {
  if (dev < 0 || dev >= kMaxDevices) return RK_ERR_CAPACITY;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || !p) return RK_ERR_CUDA;
    g_addr[dev] = p;
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
    char* w = static_cast<char*>(base);
    a.ws_o = reinterpret_cast<float*>(w);
    size_t off = static_cast<size_t>(p->num_parts) * kSplitHeads * p->d_v * sizeof(float);
    a.ws_lse = reinterpret_cast<float*>(w + off);
    off += static_cast<size_t>(p->num_parts) * kSplitHeads * sizeof(float);
    off = (off + 255) & ~size_t(255);
    a.ws_ticket = reinterpret_cast<int32_t*>(w + off);
    if (cudaMemsetAsync(a.ws_ticket, 0, p->num_mgroups * sizeof(int32_t), s) != cudaSuccess)
      return RK_ERR_CUDA;
  }
  return rk::launch_forward(*p, a, q, s) == cudaSuccess ? RK_OK : RK_ERR_CUDA;
}
