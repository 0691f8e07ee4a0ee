// fa_bwd_noalloc: the backward pass for callers that cannot allocate device
// memory.
//
// fa_bwd needs a device workspace (D, the base-2 LSE and an fp32 dQ
// accumulator) that the caller allocates. Some callers have no way to do
// that while attention runs: a runtime that plans all device memory up
// front and hands kernels only the input and output buffers; code that runs
// inside an allocator or memory-pool callback, where calling the allocator
// again would re-enter it; latency-bound services that may not call
// cudaMalloc on the request path because it can synchronise the device and
// has no latency bound. For them this entry point takes the workspace from a
// fixed array in device memory that the library itself declares, so the call
// allocates nothing.
//
// Cost and limits:
//  - the array (FA_NOALLOC_SCRATCH_BYTES, 32 MiB) is part of the library's
//    device image: every GPU on which the library is loaded holds it until
//    the process exits;
//  - problems whose workspace (fa_bwd_workspace_size) exceeds it are rejected
//    with FA_ERR_UNSUPPORTED before anything is launched;
//  - all calls share the one array, so calls whose work overlaps on the GPU
//    (different streams, different host threads) race and give wrong results;
//    serialise them. The array keeps whatever the last call left in it; that
//    does not matter, because the first launch of the backward rewrites every
//    part of the workspace it later reads (it zeroes the dQ accumulator).
//  - the first call on each device looks up the array's device address
//    (cudaGetSymbolAddress, with that device current) and caches it with the
//    id of the device's context; make that first call before any stream
//    capture. After cudaDeviceReset the device gets a new context (and the
//    array a new address): the next call sees the new id and looks the
//    address up again, so it too should come before any capture.
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "fa.h"
#include "fa_internal.h"

namespace {

static __device__ __align__(256) unsigned char g_fa_noalloc_scratch[FA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices];
unsigned long long g_scratch_ctx[kMaxDevices];   // context id each address belongs to

// Device address of the scratch array on the current device (looked up once
// per device and context; in host code the array's name is only a host-side
// stand-in).
fa_status scratch_on_current_device(void** out) {
  int dev = 0;
  unsigned long long ctx = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FA_ERR_CUDA;
  if (fa::current_context_id(&ctx) != FA_OK) return FA_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (!g_scratch_addr[dev] || g_scratch_ctx[dev] != ctx) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_fa_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr) return FA_ERR_CUDA;
    g_scratch_addr[dev] = p;
    g_scratch_ctx[dev] = ctx;
  }
  *out = g_scratch_addr[dev];
  return FA_OK;
}

}  // namespace

extern "C" fa_status fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o,
                                    const float* lse, const void* dO, void* dq, void* dk,
                                    void* dv, const float* key_bias, int B, int H, int Nq,
                                    int Nk, int d, float scale, int causal, fa_dtype dtype,
                                    void* stream) {
  const size_t need = fa_bwd_workspace_size(B, H, Nq, Nk, d);
  if (need == 0) return FA_ERR_INVALID_ARG;
  if (need > (size_t)FA_NOALLOC_SCRATCH_BYTES) return FA_ERR_UNSUPPORTED;
  void* ws = nullptr;
  const fa_status st = scratch_on_current_device(&ws);
  if (st != FA_OK) return st;
  return fa_bwd(q, k, v, o, lse, dO, dq, dk, dv, key_bias, B, H, Nq, Nk, d, scale, causal, dtype,
                ws, (size_t)FA_NOALLOC_SCRATCH_BYTES, stream);
}
