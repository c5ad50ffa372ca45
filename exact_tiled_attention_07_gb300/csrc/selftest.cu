// Self-test of the bounded waits: a CTA waits on an mbarrier phase that nothing completes (or,
// as the control case, that its own thread completes), with a short limit.  The wait gives
// up, records a timeout in the device error word and the kernel returns, so the context stays
// usable; fa_check_device_error then reports FA_ERR_TIMEOUT.  Every kernel of the library
// waits through the same mbar_wait_for.
#include <cuda_runtime.h>
#include <cstdint>

#include "kernels.h"
#include "ptx.cuh"

namespace fa {
namespace {

constexpr uint32_t kSelftestSite = 900;
constexpr uint32_t kDebugCheckSite = 901;

// One index check of the kind debug builds make inside the kernels (debug_check): out of
// [0, limit) it is recorded as a failed device check at site 901.
__global__ void debug_check_selftest_kernel(unsigned long long* err, int index, int limit) {
  __shared__ int abort_flag;
  abort_flag = 0;
  const ErrCtx ctx{err, &abort_flag};
  debug_check(index >= 0 && index < limit, ctx, kDebugCheckSite);
}

__global__ void bounded_wait_selftest_kernel(unsigned long long* err, uint64_t limit_ns, int arrive) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (arrive && threadIdx.x == 0) mbar_arrive(&bar);
  const ErrCtx ctx{err, &abort_flag};
  mbar_wait_for(&bar, 0, ctx, kSelftestSite, limit_ns);
}

// One reading per SM of its cycle counter (%clock64, SM clock cycles, free-running across
// kernels) and of the global nanosecond timer.  Each block asks for more shared memory than two
// blocks can share, so a grid of one block per SM puts one block on every idle SM.  Two
// readings taken around a stretch of work give each SM's mean clock over it.
constexpr int kClockSampleSmem = 160 * 1024;

__global__ void sm_clock_sample_kernel(unsigned long long* out) {
  extern __shared__ uint8_t pad[];
  if (threadIdx.x == 0) {
    uint32_t smid;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
    pad[0] = (uint8_t)smid;  // keeps the shared allocation
    const unsigned long long c = clock64();
    const unsigned long long t = globaltimer();
    out[3 * blockIdx.x] = smid;
    out[3 * blockIdx.x + 1] = c;
    out[3 * blockIdx.x + 2] = t;
  }
}

}  // namespace

cudaError_t launch_sm_clock_sample(unsigned long long* out, int blocks, cudaStream_t stream) {
  cudaError_t e = cudaFuncSetAttribute(sm_clock_sample_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kClockSampleSmem);
  if (e != cudaSuccess) return e;
  sm_clock_sample_kernel<<<blocks, 32, kClockSampleSmem, stream>>>(out);
  return cudaGetLastError();
}

cudaError_t launch_debug_check_selftest(unsigned long long* err, int index, int limit, cudaStream_t stream) {
  debug_check_selftest_kernel<<<1, 1, 0, stream>>>(err, index, limit);
  return cudaGetLastError();
}

cudaError_t launch_bounded_wait_selftest(unsigned long long* err, int timeout_ms, int arrive, cudaStream_t stream) {
  bounded_wait_selftest_kernel<<<1, 32, 0, stream>>>(err, (uint64_t)timeout_ms * 1000000ull, arrive);
  return cudaGetLastError();
}

}  // namespace fa
