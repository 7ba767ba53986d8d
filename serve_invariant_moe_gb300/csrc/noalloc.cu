// noalloc.cu -- moe_route_topk without a caller-provided workspace.
//
// moe_route_topk needs a little device scratch besides its inputs and outputs:
// the status word, the dynamic-schedule counter of the router GEMM, and one
// count per (64-token chunk, expert) for the deterministic counting sort.  The
// regular entry point takes that scratch as a workspace the caller allocates.
// Some callers cannot allocate device memory at the point where they route
// tokens -- for example a serving loop that runs under a fixed memory budget
// and may not call cudaMalloc there (it can fail under pressure and it
// synchronises the device), or a plain-C host that only holds the buffers it
// was handed.  For them this file keeps the scratch in one fixed device array
// that lives as long as the library is loaded.
#include <cuda_runtime.h>

#include <mutex>

#include "internal.h"

namespace invmoe {

namespace {

// 256 bytes of status block (status word, schedule counter) + 1 MiB of chunk counts.
constexpr size_t kNoAllocCountBytes = size_t(1) << 20;
constexpr size_t kNoAllocBytes = kStatusBytes + kNoAllocCountBytes;

// One copy per device that loads the library; every call on that device shares it.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocBytes];

// Device address of g_noalloc_scratch, looked up once per device with that
// device current.  In host code the symbol itself is only a host-side handle,
// so it must never be passed to a kernel directly.  The cached address belongs
// to the device's primary context at the time of the lookup; a device reset
// replaces that context (and the module holding the array), so the entry point
// is not for use after one (the header says so).
std::mutex g_noalloc_mu;
void* g_noalloc_ptr[64] = {};

int noalloc_scratch(void** out) {
  int dev = 0;
  int rc = check_cuda(cudaGetDevice(&dev), "cudaGetDevice");
  if (rc) return rc;
  if (dev < 0 || dev >= 64) return set_error(INVMOE_ERR_UNSUPPORTED_SHAPE, "device index %d out of range", dev);
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (g_noalloc_ptr[dev] == nullptr) {
    void* p = nullptr;
    rc = check_cuda(cudaGetSymbolAddress(&p, g_noalloc_scratch), "cudaGetSymbolAddress(g_noalloc_scratch)");
    if (rc) return rc;
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return INVMOE_OK;
}

}  // namespace

}  // namespace invmoe

using namespace invmoe;

extern "C" int moe_route_topk_noalloc(const void* x, const void* w_router, int T, int H, int E, int k,
                                      float* logits, int32_t* topk_idx, float* topk_w, int32_t* plan, void* xp,
                                      unsigned int* status, void* stream) {
  if (T < 0 || H <= 0 || E <= 0 || k <= 0)
    return set_error(INVMOE_ERR_INVALID_ARG, "need T >= 0, H, E, k > 0");
  if (E > 1024) return set_error(INVMOE_ERR_UNSUPPORTED_SHAPE, "E=%d > 1024", E);
  if (k > E || k > 32) return set_error(INVMOE_ERR_INVALID_ARG, "need k <= min(E, 32) (k=%d, E=%d)", k, E);
  const size_t nc = (static_cast<size_t>(T) + kDispatchChunk - 1) / kDispatchChunk;
  if (nc * static_cast<size_t>(E) * sizeof(int32_t) > kNoAllocCountBytes)
    return set_error(INVMOE_ERR_UNSUPPORTED_SHAPE,
                     "T=%d, E=%d exceed the fixed scratch of moe_route_topk_noalloc: need ceil(T/64)*E <= %zu",
                     T, E, kNoAllocCountBytes / sizeof(int32_t));
  if (status != nullptr && (reinterpret_cast<uintptr_t>(status) & 3u) != 0)
    return set_error(INVMOE_ERR_MISALIGNED, "status is not 4-byte aligned");
  void* scratch = nullptr;
  int rc = noalloc_scratch(&scratch);
  if (rc) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // the status word must start at zero (the schedule counters start at zero in the static array and
  // every GEMM launch leaves them at zero)
  rc = check_cuda(cudaMemsetAsync(scratch, 0, sizeof(unsigned int), st), "cudaMemsetAsync");
  if (rc) return rc;
  // Same validation and the same kernels as moe_route_topk, on the fixed scratch.
  rc = moe_route_topk(x, w_router, T, H, E, k, logits, topk_idx, topk_w, plan, xp, scratch, kNoAllocBytes, stream);
  if (rc) return rc;
  if (status != nullptr)
    rc = check_cuda(cudaMemcpyAsync(status, scratch, sizeof(unsigned int), cudaMemcpyDeviceToDevice, st),
                    "cudaMemcpyAsync");
  return rc;
}
