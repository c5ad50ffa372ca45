// FP8 (E4M3) block quantisation.
//
// "Lecture 8 · GPU Performance & FlashAttention" §8.1 and "FlashAttention and GPU memory" §11:
// the third generation runs attention in 8-bit floating point with block quantisation, one
// scale per block of each tensor.  Here a block is 128 rows x d of one head (the tile the
// forward streams), its scale is amax / 448 (E4M3's largest finite value) and its codes are
// E4M3(x / scale), rounded to nearest even; the scale and the quotient are fp32 divisions.
// The FP8 forward itself is the 16-bit forward's kernel with 8-bit operands (fwd_tc.cu, F8).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <algorithm>
#include <cmath>
#include <cstdint>

#include "kernels.h"
#include "ptx.cuh"
#include "tmap.h"

namespace fa {
namespace {

constexpr float kE4m3Max = 448.0f;

// ------------------------------------------------------------------------------ quantisation

// 8 consecutive elements as raw words (16-bit types: one 16-byte load; fp32: two), and their
// fp32 values
template <typename T>
struct Raw8 {
  static constexpr int W = sizeof(T) == 4 ? 8 : 4;  // 32-bit words
  uint32_t w[W];
};
template <typename T>
__device__ __forceinline__ void load_raw8(const T* p, Raw8<T>& r) {
  const uint4* q = reinterpret_cast<const uint4*>(p);
#pragma unroll
  for (int i = 0; i < Raw8<T>::W / 4; ++i) {
    const uint4 u = q[i];
    r.w[4 * i] = u.x;
    r.w[4 * i + 1] = u.y;
    r.w[4 * i + 2] = u.z;
    r.w[4 * i + 3] = u.w;
  }
}
__device__ __forceinline__ void unpack8f(const Raw8<float>& r, float (&x)[8]) {
#pragma unroll
  for (int i = 0; i < 8; ++i) x[i] = __uint_as_float(r.w[i]);
}
__device__ __forceinline__ void unpack8f(const Raw8<__nv_bfloat16>& r, float (&x)[8]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    x[2 * i] = __uint_as_float(r.w[i] << 16);
    x[2 * i + 1] = __uint_as_float(r.w[i] & 0xFFFF0000u);
  }
}
__device__ __forceinline__ void unpack8f(const Raw8<__half>& r, float (&x)[8]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&r.w[i]));
    x[2 * i] = f.x;
    x[2 * i + 1] = f.y;
  }
}

// Codes of 8 quotients v / s, bit for bit those of the correctly rounded fp32 quotients.
// q = v * (1/s) is within 2^-21 |q| of fp32(v / s); rounding to E4M3 is monotonic, so when
// q (1 - 2^-20) and q (1 + 2^-20) give the same code, that is the code of fp32(v / s).  Only a
// group with a quotient that close to an E4M3 rounding boundary divides exactly.
__device__ __forceinline__ uint2 e4m3_codes8(const float (&v)[8], float s, float rs) {
  constexpr float kLo = 1.0f - 0x1p-20f, kHi = 1.0f + 0x1p-20f;
  float lo[8], hi[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float q = v[i] * rs;
    lo[i] = q * kLo;
    hi[i] = q * kHi;
  }
  uint2 c = make_uint2(pack4_e4m3(lo[0], lo[1], lo[2], lo[3]), pack4_e4m3(lo[4], lo[5], lo[6], lo[7]));
  const uint2 h = make_uint2(pack4_e4m3(hi[0], hi[1], hi[2], hi[3]), pack4_e4m3(hi[4], hi[5], hi[6], hi[7]));
  if ((c.x != h.x) | (c.y != h.y)) {
    float q[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) q[i] = __fdiv_rn(v[i], s);
    c = make_uint2(pack4_e4m3(q[0], q[1], q[2], q[3]), pack4_e4m3(q[4], q[5], q[6], q[7]));
  }
  return c;
}

// One CTA per 128-row block of one head (fp32 inputs): amax over the block, then the codes; the
// block stays in registers as the input's raw words and is unpacked twice.
template <typename T, int D>
__global__ void __launch_bounds__(256) quantize_fp8_kernel(const T* __restrict__ x, uint8_t* __restrict__ x8,
                                                           float* __restrict__ scales, int n, int nb) {
  constexpr int G = 128 * D / 8 / 256;  // 8-element groups per thread in a full block
  __shared__ float red[8];
  const int blk = blockIdx.x % nb;
  const int64_t head = blockIdx.x / nb;
  const int r0 = blk * 128;
  const int groups = min(128, n - r0) * D / 8;
  const T* src = x + (head * n + r0) * D;
  uint8_t* dst = x8 + (head * n + r0) * D;
  Raw8<T> raw[G];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    const int gi = threadIdx.x + g * 256;
    if (gi < groups) {
      load_raw8(src + (int64_t)gi * 8, raw[g]);
    } else {
#pragma unroll
      for (int i = 0; i < Raw8<T>::W; ++i) raw[g].w[i] = 0u;
    }
  }
  float amax = 0.f;
#pragma unroll
  for (int g = 0; g < G; ++g) {
    float v[8];
    unpack8f(raw[g], v);
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
  }
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
  __syncthreads();
  amax = red[0];
#pragma unroll
  for (int w = 1; w < 8; ++w) amax = fmaxf(amax, red[w]);
  const float s = amax > 0.f ? __fdiv_rn(amax, kE4m3Max) : 1.f;
  const float rs = __frcp_rn(s);
  if (threadIdx.x == 0) scales[head * nb + blk] = s;
#pragma unroll
  for (int g = 0; g < G; ++g) {
    const int gi = threadIdx.x + g * 256;
    if (gi < groups) {
      float v[8];
      unpack8f(raw[g], v);
      *reinterpret_cast<uint2*>(dst + (int64_t)gi * 8) = e4m3_codes8(v, s, rs);
    }
  }
}

// Streaming variant for 16-bit inputs.  A 128-row block of one head is contiguous in memory,
// so a persistent grid walks the blocks and one thread pulls each into a two-stage
// shared-memory ring with a single bulk copy: the next block lands while the current one is
// quantised (the register variant above keeps loads in flight only between a block's start and
// its reduction).  Every thread runs every iteration and reaches every __syncthreads; a thread
// whose bounded wait ran out skips the work.
// |x| maxima of 8 16-bit values as their bit patterns: for non-negative floats these order as
// unsigned integers, so two per instruction
template <typename T>
__device__ __forceinline__ uint32_t absmax_bits(const Raw8<T>& r, uint32_t m) {
  static_assert(sizeof(T) == 2, "16-bit inputs");
#pragma unroll
  for (int i = 0; i < 4; ++i) m = __vmaxu2(m, r.w[i] & 0x7FFF7FFFu);
  return m;
}
__device__ __forceinline__ float bits16_to_float(uint32_t b, const __nv_bfloat16*) { return __uint_as_float(b << 16); }
__device__ __forceinline__ float bits16_to_float(uint32_t b, const __half*) {
  return __half2float(__ushort_as_half((unsigned short)b));
}

template <typename T, int D>
__global__ void __launch_bounds__(256) quantize_fp8_stream(const T* __restrict__ x, uint8_t* __restrict__ x8,
                                                           float* __restrict__ scales, int n, int nb, int64_t total,
                                                           unsigned long long* err) {
  static_assert(sizeof(T) == 2, "16-bit inputs");
  constexpr int BLK = 128 * D * 2;      // bytes of a full block
  constexpr int G = 128 * D / 8 / 256;  // 8-element groups per thread in a full block
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + 2 * BLK);  // [2]
  float* red = reinterpret_cast<float*>(full + 2);                // [8]
  volatile int* abort_flag = reinterpret_cast<volatile int*>(red + 8);
  const ErrCtx ctx{err, abort_flag};
  if (threadIdx.x == 0) {
    *abort_flag = 0;
    mbar_init(full, 1);
    mbar_init(full + 1, 1);
    fence_barrier_init();
  }
  __syncthreads();
  const int64_t first = blockIdx.x, step = gridDim.x;
  auto rows_of = [&](int64_t b) { return min(128, n - (int)(b % nb) * 128); };
  // block b -> stage s (thread 0)
  auto issue = [&](int64_t b, int s) {
    const int64_t head = b / nb;
    const int r0 = (int)(b % nb) * 128;
    const uint32_t bytes = (uint32_t)rows_of(b) * D * 2;
    mbar_arrive_expect_tx(full + s, bytes);
    bulk_load(smem + s * BLK, x + (head * n + r0) * D, bytes, full + s);
  };
  if (threadIdx.x == 0) {
    if (first < total) issue(first, 0);
    if (first + step < total) issue(first + step, 1);
  }
  bool ok = true;
  int it = 0;
  for (int64_t b = first; b < total; b += step, ++it) {
    const int s = it & 1;
    ok = mbar_wait(full + s, (uint32_t)(it >> 1) & 1, ctx, 60) && ok;
    const int64_t head = b / nb;
    const int blk = (int)(b % nb);
    const int groups = rows_of(b) * D / 8;
    const Raw8<T>* src = reinterpret_cast<const Raw8<T>*>(smem + s * BLK);
    uint32_t mb = 0u;
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const int gi = threadIdx.x + g * 256;
      if (ok && gi < groups) mb = absmax_bits(src[gi], mb);
    }
    float amax = bits16_to_float(max(mb & 0xFFFFu, mb >> 16), static_cast<const T*>(nullptr));
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
    __syncthreads();
    amax = red[0];
#pragma unroll
    for (int w = 1; w < 8; ++w) amax = fmaxf(amax, red[w]);
    const float sc = amax > 0.f ? __fdiv_rn(amax, kE4m3Max) : 1.f;
    const float rs = __frcp_rn(sc);
    if (threadIdx.x == 0 && ok) scales[head * nb + blk] = sc;
    uint8_t* dst = x8 + (head * n + blk * 128) * D;
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const int gi = threadIdx.x + g * 256;
      if (ok && gi < groups) {
        float v[8];
        unpack8f(src[gi], v);
        *reinterpret_cast<uint2*>(dst + (int64_t)gi * 8) = e4m3_codes8(v, sc, rs);
      }
    }
    __syncthreads();  // stage s read by every thread, and red free again
    if (threadIdx.x == 0 && b + 2 * step < total) issue(b + 2 * step, s);
  }
  // a copy whose wait ran out may still be in flight: it must land before the CTA exits
  if (threadIdx.x == 0 && !ok) {
    ErrCtx nctx = ctx;
    int no_abort = 0;
    nctx.abort = &no_abort;
    for (int j = it - 1; j >= 0 && j >= it - 2; --j) mbar_wait(full + (j & 1), (uint32_t)(j >> 1) & 1, nctx, 61);
  }
}

template <typename T, int D>
cudaError_t launch_quantize_stream(const QuantArgs& a, int nb) {
  constexpr int BLK = 128 * D * 2;
  const int smem = 2 * BLK + 2 * 8 + 8 * 4 + 16;
  auto kern = quantize_fp8_stream<T, D>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int64_t total = (int64_t)a.bh * nb;
  const int per_sm = std::max(1, std::min(4, 200 * 1024 / smem));
  const int64_t grid = std::min<int64_t>(total, (int64_t)device_sm_count() * per_sm);
  kern<<<(unsigned)grid, 256, smem, a.stream>>>((const T*)a.x, (uint8_t*)a.x8, a.scales, a.n, nb, total, a.err);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_quantize_t(const QuantArgs& a) {
  const int nb = (a.n + 127) / 128;
  if constexpr (sizeof(T) == 2) {
    switch (a.d) {
      case 64: return launch_quantize_stream<T, 64>(a, nb);
      case 128: return launch_quantize_stream<T, 128>(a, nb);
      case 256: return launch_quantize_stream<T, 256>(a, nb);
      default: return cudaErrorNotSupported;
    }
  } else {
    const unsigned grid = (unsigned)((int64_t)a.bh * nb);
    switch (a.d) {
      case 64:
        quantize_fp8_kernel<T, 64><<<grid, 256, 0, a.stream>>>((const T*)a.x, (uint8_t*)a.x8, a.scales, a.n, nb);
        break;
      case 128:
        quantize_fp8_kernel<T, 128><<<grid, 256, 0, a.stream>>>((const T*)a.x, (uint8_t*)a.x8, a.scales, a.n, nb);
        break;
      case 256:
        quantize_fp8_kernel<T, 256><<<grid, 256, 0, a.stream>>>((const T*)a.x, (uint8_t*)a.x8, a.scales, a.n, nb);
        break;
      default:
        return cudaErrorNotSupported;
    }
    return cudaGetLastError();
  }
}

}  // namespace

cudaError_t launch_quantize_fp8(const QuantArgs& a) {
  switch (a.dtype) {
    case DT_BF16: return launch_quantize_t<__nv_bfloat16>(a);
    case DT_FP16: return launch_quantize_t<__half>(a);
    default: return launch_quantize_t<float>(a);
  }
}

}  // namespace fa
