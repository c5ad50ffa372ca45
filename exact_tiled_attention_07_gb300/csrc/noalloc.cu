// fa_bwd_noalloc: the backward pass with its scratch in a fixed device array, for callers
// that must not allocate device memory themselves.
//
// fa_bwd needs a caller-provided workspace (per head: D, L*log2 e and an fp32 dQ
// accumulator).  Some callers cannot get one: code that runs inside a host application
// which owns every device allocation (a plugin or runtime with its own memory pool, where
// an extra cudaMalloc would bypass that pool's accounting), or a latency-bound loop where
// cudaMalloc's implicit device synchronisation is not acceptable.  For them this entry
// point uses a file-scope __device__ array as the workspace instead; the caller still
// passes every input and output.
//
// The array is part of this library's device image, so every GPU on which the library
// is loaded holds it (FA_BWD_NOALLOC_SCRATCH_BYTES) until the process exits.  All calls
// share it: two calls whose kernels overlap on the GPU (other streams, other host threads)
// race on it.  Each call rewrites everything it reads from it (the preprocess kernel
// writes D and L*log2 e and zeroes the dQ accumulator), so no state leaks between calls.
#include <cuda_runtime.h>
#include <cstdint>
#include <mutex>

#include "fa.h"
#include "kernels.h"

namespace fa {
namespace {

__device__ __align__(256) unsigned char g_bwd_scratch[FA_BWD_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
struct ScratchAddr {
  void* ptr = nullptr;
  unsigned long long ctx = 0;  // id of the context the address belongs to
};
ScratchAddr g_scratch_addr[kMaxDevices];
std::mutex g_scratch_mu;

// Device address of g_bwd_scratch on the current device.  In host code the array's name
// is only a host-side stand-in; the address comes from cudaGetSymbolAddress, looked up with
// the device current on the first call in each context (once per device, unless the device's
// context is destroyed and recreated, e.g. by cudaDeviceReset, when it is looked up again).
fa_status scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return (fa_status)set_last_error(FA_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices)
    return (fa_status)set_last_error(FA_ERR_UNSUPPORTED, "device index %d out of range", dev);
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  ScratchAddr& a = g_scratch_addr[dev];
  const unsigned long long ctx = current_context_id();
  if (!a.ptr || ctx == 0 || ctx != a.ctx) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_bwd_scratch);
    if (e != cudaSuccess || !p)
      return (fa_status)set_last_error(FA_ERR_CUDA, "cudaGetSymbolAddress(backward scratch): %s",
                                       cudaGetErrorString(e));
    a.ptr = p;
    a.ctx = current_context_id();  // the lookup made the device's context current if none was
  }
  *out = a.ptr;
  return FA_OK;
}

}  // namespace
}  // namespace fa

extern "C" fa_status fa_bwd_noalloc(const void* Q, const void* K, const void* V, const void* O, const void* dO,
                                    const float* L, void* dQ, void* dK, void* dV, int B, int H, int N, int d,
                                    float scale, int causal, fa_dtype dtype, void* stream) {
  const size_t need = fa_bwd_workspace_size(B, H, N, d);
  if (need == 0 && (int64_t)B * H * N != 0)
    return (fa_status)fa::set_last_error(FA_ERR_INVALID_ARG, "fa_bwd_noalloc: invalid sizes B=%d H=%d N=%d d=%d", B,
                                         H, N, d);
  if (need > (size_t)FA_BWD_NOALLOC_SCRATCH_BYTES)
    return (fa_status)fa::set_last_error(FA_ERR_INVALID_ARG,
                                         "fa_bwd_noalloc: B=%d H=%d N=%d d=%d needs %zu bytes of scratch, more than "
                                         "the %llu-byte static array; use fa_bwd with a workspace",
                                         B, H, N, d, need, (unsigned long long)FA_BWD_NOALLOC_SCRATCH_BYTES);
  void* scratch = nullptr;
  fa_status st = fa::scratch_address(&scratch);
  if (st != FA_OK) return st;
  return fa_bwd(Q, K, V, O, dO, L, dQ, dK, dV, scratch, (size_t)FA_BWD_NOALLOC_SCRATCH_BYTES, B, H, N, d, scale,
                causal, dtype, stream);
}
