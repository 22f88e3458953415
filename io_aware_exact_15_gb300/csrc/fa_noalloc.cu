// fa_backward_noalloc: the backward pass for callers that cannot allocate
// device memory.  Its scratch (the D vector and the fp32 dQ accumulator that
// fa_backward takes as a caller-owned workspace) lives in one fixed-size
// file-scope device array instead.
//
// Who needs this: code that runs inside a host framework that hands out no
// workspace (a plugin or callback interface with no workspace query), and
// code that must not call cudaMalloc once it is running, because cudaMalloc
// can synchronise the device, can fail under memory pressure in the middle
// of a job, and is not available to it at all inside some runtimes.
//
// Costs and rules:
//  * every GPU that loads this library holds kNoAllocScratchBytes of device
//    memory for the array until the process exits;
//  * problems whose workspace exceeds that size are rejected with
//    FA_ERR_WORKSPACE before anything is launched;
//  * all calls on a device share the one array and it keeps the previous
//    call's contents; the preprocess kernel rewrites D and zeroes the dQ
//    accumulator at the start of every call, so stale contents never leak
//    into a result, but two calls whose kernels overlap on the GPU (different
//    streams, no ordering between them) race on the array;
//  * the first call on each device looks up the array's device address
//    (cudaGetSymbolAddress, with that device current) and caches it; make
//    that first call before any stream capture.
#include <atomic>
#include <mutex>

#include "../../include/fa.h"

namespace {
constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;  // 32 MiB per device
}

// Host code must not use this name as an address: on the host it is only a
// stand-in for the device symbol.  The device address comes from
// cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_fa_noalloc_scratch[kNoAllocScratchBytes];

namespace {

constexpr int kMaxDevices = 64;
std::atomic<void*> g_scratch_addr[kMaxDevices];
std::mutex g_scratch_mu;

// Device address of the scratch array on the current device (looked up once
// per device and cached).
fa_status scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FA_ERR_CUDA;
  void* p = g_scratch_addr[dev].load();
  if (!p) {
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    p = g_scratch_addr[dev].load();
    if (!p) {
      if (cudaGetSymbolAddress(&p, g_fa_noalloc_scratch) != cudaSuccess || !p) return FA_ERR_CUDA;
      g_scratch_addr[dev].store(p);
    }
  }
  *out = p;
  return FA_OK;
}

}  // namespace

extern "C" fa_status fa_backward_noalloc(const void* q, const void* k, const void* v,
                                         const void* o, const void* dO, const float* lse,
                                         void* dq, void* dk, void* dv, int B, int H, int N, int d,
                                         float scale, int causal, cudaStream_t stream) {
  const size_t need = fa_backward_workspace_size(B, H, N, d);
  if (need == 0) return FA_ERR_INVALID_ARG;
  if (need > kNoAllocScratchBytes) return FA_ERR_WORKSPACE;
  void* scratch = nullptr;
  const fa_status st = scratch_address(&scratch);
  if (st != FA_OK) return st;
  return fa_backward(q, k, v, o, dO, lse, dq, dk, dv, B, H, N, d, scale, causal, scratch,
                     kNoAllocScratchBytes, stream);
}
