// noalloc.cu -- a dispatch entry point that needs no workspace.
//
// Some callers cannot hand this library a workspace: a serving runtime that
// reserves all of HBM for weights and KV cache when it starts and gives out
// no further buffers, plain C code that links only this library and has no
// device allocator of its own, or code running where a cudaMalloc would be
// unsafe or forbidden (inside a memory pool that must not grow, or on a path
// that must not synchronise the device, which cudaMalloc/cudaFree can do).
// moe_dispatch_noalloc serves them: the per-chunk expert histograms that
// moe_dispatch keeps in the caller's workspace live here in one file-scope
// device array instead, of a fixed size.
//
// Every GPU that loads this library holds the array until the process
// exits.  All calls on a device share it, so two calls that overlap on the
// GPU (different streams, no ordering between them) race on it; calls on
// one stream, or otherwise ordered, are safe.  Each call overwrites every
// entry it reads, so nothing needs clearing between calls.
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace {

// chunks * E int32 histograms; 1 MiB.
constexpr int64_t kNoAllocScratchInts = 262144;
static __device__ __align__(256) int32_t g_dispatch_scratch[kNoAllocScratchInts];

constexpr int kMaxDevices = 64;

// cuCtxGetCurrent / cuCtxGetId of the driver, looked up through the runtime
// (the library does not link libcuda).  A context's id is never reused, so
// a cached address is known to belong to the context that is current now.
struct CtxApi {
  int (*get_current)(void **ctx) = nullptr;
  int (*get_id)(void *ctx, unsigned long long *id) = nullptr;
};

const CtxApi &ctx_api() {
  static const CtxApi api = [] {
    CtxApi a;
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      a.get_current = reinterpret_cast<int (*)(void **)>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      a.get_id = reinterpret_cast<int (*)(void *, unsigned long long *)>(p);
    return a;
  }();
  return api;
}

bool current_ctx_id(unsigned long long *id) {
  const CtxApi &api = ctx_api();
  void *ctx = nullptr;
  return api.get_current && api.get_id && api.get_current(&ctx) == 0 && ctx != nullptr &&
         api.get_id(ctx, id) == 0;
}

struct ScratchAddr {
  unsigned long long ctx_id = 0;
  int32_t *addr = nullptr;
};
std::mutex g_scratch_mu;
ScratchAddr g_scratch_addr[kMaxDevices];

// Device address of the array in the current device's context.  In host
// code the array's name is only a host-side stand-in, so the address is
// looked up with the device current -- on the first call on a device, and
// again whenever that device's context has changed (after a
// cudaDeviceReset the module is loaded anew, possibly elsewhere) -- and
// cached with the id of the context it belongs to.
moe_status_t scratch_address(int32_t **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return MOE_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  unsigned long long id = 0;
  ScratchAddr &c = g_scratch_addr[dev];
  if (!current_ctx_id(&id) || c.addr == nullptr || c.ctx_id != id) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_dispatch_scratch) != cudaSuccess || p == nullptr)
      return MOE_ERR_CUDA;
    // the lookup has made the device's primary context current if it was not
    if (!current_ctx_id(&id)) return MOE_ERR_CUDA;
    c.ctx_id = id;
    c.addr = static_cast<int32_t *>(p);
  }
  *out = c.addr;
  return MOE_OK;
}

}  // namespace

extern "C" moe_status_t moe_dispatch_noalloc(const moe_shape_t *shape, const int32_t *topk_ids,
                                              const void *x, int32_t *counts, int32_t *offsets,
                                              int32_t *src_token, int32_t *dest, void *x_perm,
                                              moe_stream_t stream) {
  const moe_status_t st = moe::check_shape_for_abi(shape);
  if (st != MOE_OK) return st;
  if (shape->T == 0) return MOE_OK;
  if (!topk_ids || !counts || !offsets || !src_token || !dest) return MOE_ERR_INVALID_ARG;
  if (x && !x_perm) return MOE_ERR_INVALID_ARG;
  if (x && ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(x_perm)) & 15u))
    return MOE_ERR_INVALID_ARG;
  const int64_t n = static_cast<int64_t>(shape->T) * shape->k;
  if (moe::dispatch_num_chunks(n) * shape->E > kNoAllocScratchInts) return MOE_ERR_UNSUPPORTED;
  int32_t *scratch = nullptr;
  const moe_status_t ast = scratch_address(&scratch);
  if (ast != MOE_OK) return ast;
  const cudaError_t err = moe::launch_dispatch(topk_ids, shape->T, shape->k, shape->E, x,
                                               shape->d, counts, offsets, src_token, dest, x_perm,
                                               scratch, nullptr, 128, nullptr, stream);
  return err == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
