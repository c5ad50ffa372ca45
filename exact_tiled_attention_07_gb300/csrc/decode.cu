// Decode attention over a long key/value cache, split across CTAs (CUDA cores, HBM-bound).
//
// A few query rows (Nq new positions, every query head of a grouped key/value head) attend
// to all Nk cached keys ("Lecture 8 · GPU Performance & FlashAttention" §8.2: the cache is
// cut into pieces processed in parallel, and the pieces are combined with the merge formula
// of the online softmax, Exercise 3).  Each step reads every cached key and value once and
// does about 2·d multiply-adds per (row, key), so with up to 8 rows per CTA the kernel is
// bound by HBM bandwidth, not by a contraction: it runs on CUDA cores with coalesced 16-byte
// loads instead of padding 8 rows up to a 128-row tensor-core tile.
//
// decode_partial: CTA = (batch row, key/value head, block of <= 8 query rows, split of the
//   cache).  Its 8 warps take interleaved 32-key chunks of the split; in each chunk a lane
//   scores one key against all rows (K row in registers, Q rows broadcast from shared
//   memory), the warp runs the online softmax per row, then lanes switch to owning head
//   dimensions and accumulate P·V with coalesced V rows.  The 8 warp states are merged in
//   shared memory.  With one split the CTA writes O and L; otherwise it writes the split's
//   normalised output and base-2 log-sum-exp to the workspace.
// decode_merge: one warp per row folds the splits: L = log-sum-exp of the split L_s,
//   O = sum_s 2^(L_s - L) O_s (the Exercise 3 merge with l folded into L).
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <cmath>
#include <cstdint>

#include "kernels.h"

namespace fa {
namespace {

constexpr int kWarps = 8;
constexpr int kRowsPerCta = 8;

__device__ __forceinline__ float warp_max(float v) {
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float ex2f(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// 8 consecutive elements at p (16-byte aligned) as fp32
__device__ __forceinline__ void load8(const float* p, float (&x)[8]) {
  const float4 a = *reinterpret_cast<const float4*>(p), b = *reinterpret_cast<const float4*>(p + 4);
  x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w; x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}
__device__ __forceinline__ void load8(const __nv_bfloat16* p, float (&x)[8]) {
  const uint4 u = *reinterpret_cast<const uint4*>(p);
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    x[2 * i] = __uint_as_float(w[i] << 16);
    x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}
__device__ __forceinline__ void load8(const __half* p, float (&x)[8]) {
  const uint4 u = *reinterpret_cast<const uint4*>(p);
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
    x[2 * i] = f.x;
    x[2 * i + 1] = f.y;
  }
}

// E consecutive elements (E in {2, 4, 8}, E * sizeof(T) bytes aligned) as fp32
template <int E>
__device__ __forceinline__ void load_row(const float* p, float (&x)[E]) {
#pragma unroll
  for (int i = 0; i < E; i += 2) {
    const float2 f = *reinterpret_cast<const float2*>(p + i);
    x[i] = f.x;
    x[i + 1] = f.y;
  }
}
template <int E, typename T>
__device__ __forceinline__ void load_row16(const T* p, float (&x)[E]) {
  uint32_t w[E / 2];
  if constexpr (E == 8) {
    const uint4 u = *reinterpret_cast<const uint4*>(p);
    w[0] = u.x; w[1] = u.y; w[2] = u.z; w[3] = u.w;
  } else if constexpr (E == 4) {
    const uint2 u = *reinterpret_cast<const uint2*>(p);
    w[0] = u.x; w[1] = u.y;
  } else {
    w[0] = *reinterpret_cast<const uint32_t*>(p);
  }
#pragma unroll
  for (int i = 0; i < E / 2; ++i) {
    float2 f;
    if constexpr (sizeof(T) == 2 && __is_same(T, __nv_bfloat16))
      f = make_float2(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xFFFF0000u));
    else
      f = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
    x[2 * i] = f.x;
    x[2 * i + 1] = f.y;
  }
}
template <int E>
__device__ __forceinline__ void load_row(const __nv_bfloat16* p, float (&x)[E]) { load_row16<E>(p, x); }
template <int E>
__device__ __forceinline__ void load_row(const __half* p, float (&x)[E]) { load_row16<E>(p, x); }

__device__ __forceinline__ void store_t(float* p, float v) { *p = v; }
__device__ __forceinline__ void store_t(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }
__device__ __forceinline__ void store_t(__half* p, float v) { *p = __float2half_rn(v); }


// Rows of one CTA: query heads kvh*group + g, positions i, for g*nq + i in [r0, r0 + 8).
template <typename T, int D>
__global__ void __launch_bounds__(kWarps * 32, (D <= 128) ? 2 : 1) decode_partial(const T* __restrict__ Q, const T* __restrict__ K,
                                                            const T* __restrict__ V, T* __restrict__ O,
                                                            float* __restrict__ L, float* __restrict__ ws_o,
                                                            float* __restrict__ ws_l, int H, int Hkv, int nq, int nk,
                                                            int splits, int row_blocks, float scale_log2) {
  constexpr int E = D / 32;  // head dims per lane in the P.V phase
  extern __shared__ float sm[];
  float* qs = sm;                                 // [8][D], scaled by tau log2 e
  float* wo = qs + kRowsPerCta * D;               // [warps][8][D] unnormalised warp outputs
  float* wm = wo + kWarps * kRowsPerCta * D;      // [warps][8] warp maxima (base 2)
  float* wl = wm + kWarps * kRowsPerCta;          // [warps][8] warp denominators
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int group = H / Hkv;
  const int rows = group * nq;
  int t = blockIdx.x;
  const int split = t % splits;
  t /= splits;
  const int rb = t % row_blocks;
  t /= row_blocks;
  const int kvh = t % Hkv, b = t / Hkv;
  const int r0 = rb * kRowsPerCta;
  const int mc = min(kRowsPerCta, rows - r0);
  const int64_t lo = (int64_t)nk * split / splits, hi = (int64_t)nk * (split + 1) / splits;
  const T* kbase = K + ((int64_t)b * Hkv + kvh) * nk * D;
  const T* vbase = V + ((int64_t)b * Hkv + kvh) * nk * D;
  auto global_row = [&](int r) {  // row index into [B][H][Nq]
    const int gr = r0 + r, g = gr / nq, i = gr - g * nq;
    return ((int64_t)b * H + (int64_t)kvh * group + g) * nq + i;
  };
  for (int idx = threadIdx.x; idx < kRowsPerCta * D; idx += blockDim.x) {
    const int r = idx / D, c = idx - r * D;
    float v = 0.f;
    if (r < mc) {
      float x[2];
      load_row<2>(Q + global_row(r) * D + (c & ~1), x);
      v = x[c & 1] * scale_log2;
    }
    qs[idx] = v;
  }
  __syncthreads();

  float m[kRowsPerCta], l[kRowsPerCta], o[kRowsPerCta][E];
#pragma unroll
  for (int r = 0; r < kRowsPerCta; ++r) {
    m[r] = -INFINITY;
    l[r] = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) o[r][e] = 0.f;
  }
  for (int64_t c0 = lo + 32 * warp; c0 < hi; c0 += 32 * kWarps) {
    // scores of this lane's key against every row (base-2 domain)
    const int64_t j = c0 + lane;
    float sc[kRowsPerCta];
#pragma unroll
    for (int r = 0; r < kRowsPerCta; ++r) sc[r] = 0.f;
    if (j < hi) {
      const T* kr = kbase + j * D;
#pragma unroll 4
      for (int c = 0; c < D; c += 8) {
        float kx[8];
        load_row<8>(kr + c, kx);
#pragma unroll
        for (int r = 0; r < kRowsPerCta; ++r) {
          if (r >= mc) break;  // CTA-uniform
          const float4 q0 = *reinterpret_cast<const float4*>(qs + r * D + c);
          const float4 q1 = *reinterpret_cast<const float4*>(qs + r * D + c + 4);
          sc[r] = fmaf(q0.x, kx[0], fmaf(q0.y, kx[1], fmaf(q0.z, kx[2], fmaf(q0.w, kx[3], sc[r]))));
          sc[r] = fmaf(q1.x, kx[4], fmaf(q1.y, kx[5], fmaf(q1.z, kx[6], fmaf(q1.w, kx[7], sc[r]))));
        }
      }
    } else {
#pragma unroll
      for (int r = 0; r < kRowsPerCta; ++r) sc[r] = -INFINITY;
    }
    // online softmax per row over this chunk (every chunk holds at least one key)
#pragma unroll
    for (int r = 0; r < kRowsPerCta; ++r) {
      if (r >= mc) break;
      const float mnew = fmaxf(m[r], warp_max(sc[r]));
      const float alpha = ex2f(m[r] - mnew);  // 0 while m is -inf
      const float p = ex2f(sc[r] - mnew);     // 0 for keys past the split
      l[r] = l[r] * alpha + warp_sum(p);
      m[r] = mnew;
      sc[r] = p;
#pragma unroll
      for (int e = 0; e < E; ++e) o[r][e] *= alpha;
    }
    // P.V: lanes own head dims [lane*E, lane*E + E); V rows read coalesced, kVB rows per batch
    // so their loads are in flight together
    constexpr int kVB = (E >= 8) ? 4 : 8;
    const int nkeys = (int)min((int64_t)32, hi - c0);
    for (int k0 = 0; k0 < nkeys; k0 += kVB) {
      float vx[kVB][E];
#pragma unroll
      for (int u = 0; u < kVB; ++u) {
        const int kk = min(k0 + u, nkeys - 1);  // clamp: rows past the split are loaded but weighted 0
        load_row<E>(vbase + (c0 + kk) * D + lane * E, vx[u]);
      }
#pragma unroll
      for (int u = 0; u < kVB; ++u) {
#pragma unroll
        for (int r = 0; r < kRowsPerCta; ++r) {
          if (r >= mc) break;
          float pk = __shfl_sync(0xffffffffu, sc[r], (k0 + u) & 31);
          if (k0 + u >= nkeys) pk = 0.f;
#pragma unroll
          for (int e = 0; e < E; ++e) o[r][e] = fmaf(pk, vx[u][e], o[r][e]);
        }
      }
    }
  }
  // merge the warps' states (the same rescaling as the split merge)
#pragma unroll
  for (int r = 0; r < kRowsPerCta; ++r) {
#pragma unroll
    for (int e = 0; e < E; ++e) wo[(warp * kRowsPerCta + r) * D + lane * E + e] = o[r][e];
    if (lane == 0) {
      wm[warp * kRowsPerCta + r] = m[r];
      wl[warp * kRowsPerCta + r] = l[r];
    }
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < mc * D; idx += blockDim.x) {
    const int r = idx / D, c = idx - r * D;
    float mt = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) mt = fmaxf(mt, wm[w * kRowsPerCta + r]);
    float den = 0.f, num = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const float mw = wm[w * kRowsPerCta + r];
      const float f = (mw == -INFINITY) ? 0.f : ex2f(mw - mt);
      den = fmaf(wl[w * kRowsPerCta + r], f, den);
      num = fmaf(wo[(w * kRowsPerCta + r) * D + c], f, num);
    }
    const int64_t gr = global_row(r);
    const float lse2 = mt + log2f(den);
    if (splits == 1) {
      store_t(O + gr * D + c, num / den);
      if (c == 0) L[gr] = lse2 * 0.6931471805599453f;
    } else {
      ws_o[(gr * splits + split) * D + c] = num / den;
      if (c == 0) ws_l[gr * splits + split] = lse2;
    }
  }
}

// One warp per row: fold the splits' (O_s, L_s) into O and L.
template <typename T, int D>
__global__ void __launch_bounds__(256) decode_merge(const float* __restrict__ ws_o, const float* __restrict__ ws_l,
                                                    T* __restrict__ O, float* __restrict__ L, int64_t rows,
                                                    int splits) {
  const int64_t row = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const float* lr = ws_l + row * splits;
  float mx = -INFINITY;
  for (int s = lane; s < splits; s += 32) mx = fmaxf(mx, lr[s]);
  mx = warp_max(mx);
  constexpr int PL = D / 32;
  float acc[PL];
#pragma unroll
  for (int e = 0; e < PL; ++e) acc[e] = 0.f;
  float den = 0.f;
  // the splits' loads are independent: unrolled so several are in flight at once
#pragma unroll 4
  for (int s = 0; s < splits; ++s) {
    const float ls = lr[s];
    const float w = (ls == -INFINITY) ? 0.f : ex2f(ls - mx);
    den += w;
    const float* os = ws_o + (row * splits + s) * D;
#pragma unroll
    for (int e = 0; e < PL; ++e) acc[e] = fmaf(w, os[lane + 32 * e], acc[e]);
  }
#pragma unroll
  for (int e = 0; e < PL; ++e) store_t(O + row * D + lane + 32 * e, acc[e] / den);
  if (lane == 0) L[row] = (mx + log2f(den)) * 0.6931471805599453f;
}

template <typename T, int D>
cudaError_t launch_decode_t(const DecodeArgs& a) {
  const int group = a.h / a.hkv;
  const int row_blocks = (group * a.nq + kRowsPerCta - 1) / kRowsPerCta;
  const int64_t ctas = (int64_t)a.b * a.hkv * row_blocks * a.splits;
  const size_t smem = sizeof(float) * (size_t)(kRowsPerCta * D + kWarps * kRowsPerCta * D + 2 * kWarps * kRowsPerCta);
  auto kern = decode_partial<T, D>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  float* ws_o = a.ws;
  const int64_t rows = (int64_t)a.b * a.h * a.nq;
  float* ws_l = a.ws ? a.ws + rows * a.splits * D : nullptr;
  kern<<<(unsigned)ctas, kWarps * 32, smem, a.stream>>>((const T*)a.q, (const T*)a.k, (const T*)a.v, (T*)a.o, a.lse,
                                                       ws_o, ws_l, a.h, a.hkv, a.nq, a.nk, a.splits, row_blocks,
                                                       a.scale * 1.4426950408889634f);
  if ((e = cudaGetLastError()) != cudaSuccess || a.splits == 1) return e;
  return launch_decode_merge(a);
}

template <typename T, int D>
cudaError_t launch_merge_t(const DecodeArgs& a) {
  const int64_t rows = (int64_t)a.b * a.h * a.nq;
  const float* ws_o = a.ws;
  const float* ws_l = a.ws + rows * a.splits * D;
  decode_merge<T, D><<<(unsigned)((rows * 32 + 255) / 256), 256, 0, a.stream>>>(ws_o, ws_l, (T*)a.o, a.lse, rows,
                                                                                  a.splits);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_merge_d(const DecodeArgs& a) {
  switch (a.d) {
    case 64: return launch_merge_t<T, 64>(a);
    case 128: return launch_merge_t<T, 128>(a);
    case 256: return launch_merge_t<T, 256>(a);
    default: return cudaErrorNotSupported;
  }
}

template <typename T>
cudaError_t launch_decode_d(const DecodeArgs& a) {
  switch (a.d) {
    case 64: return launch_decode_t<T, 64>(a);
    case 128: return launch_decode_t<T, 128>(a);
    case 256: return launch_decode_t<T, 256>(a);
    default: return cudaErrorNotSupported;
  }
}

}  // namespace

int decode_auto_splits(int b, int h, int hkv, int nq, int nk) {
  const int64_t rb = ((int64_t)(h / hkv) * nq + kRowsPerCta - 1) / kRowsPerCta;
  const int64_t base = (int64_t)b * hkv * rb;
  // about two full waves of two CTAs per SM on a 152-SM GB300, rounded down so the last wave
  // is not a small remainder
  const int64_t target = 4 * kSmCount;
  int64_t s = target / base;
  s = std::min<int64_t>(s, (nk + 255) / 256);  // at least ~256 keys per split
  s = std::min<int64_t>(std::max<int64_t>(s, 1), 128);
  return (int)s;
}

size_t decode_workspace_bytes(int b, int h, int nq, int d, int splits) {
  if (splits <= 1) return 0;
  return (size_t)b * h * nq * splits * (d + 1) * sizeof(float);
}

cudaError_t launch_decode(const DecodeArgs& a) {
  switch (a.dtype) {
    case DT_BF16: return launch_decode_d<__nv_bfloat16>(a);
    case DT_FP16: return launch_decode_d<__half>(a);
    default: return launch_decode_d<float>(a);
  }
}

cudaError_t launch_decode_merge(const DecodeArgs& a) {
  switch (a.dtype) {
    case DT_BF16: return launch_merge_d<__nv_bfloat16>(a);
    case DT_FP16: return launch_merge_d<__half>(a);
    default: return launch_merge_d<float>(a);
  }
}

}  // namespace fa
