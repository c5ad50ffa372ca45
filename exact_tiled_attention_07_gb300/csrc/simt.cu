// CUDA-core (SIMT) kernels, computing in fp32 for every input dtype:
//   * fwd_simt      tiled forward with online softmax (true fp32 path; also any d <= 256)
//   * bwd_dkdv_simt / bwd_dq_simt   recomputing backward without atomics
//   * bwd_pre       D_i = sum_k dO_ik O_ik, L2_i = L_i log2(e), zeroed dQ accumulator
//   * dq_convert    dQ = tau * dQ_acc in the input dtype
//
// The forward follows the FA2 loop order ("Lecture 8 · GPU Performance &
// FlashAttention" §8.1; "Stanford CS336 Lecture 5 close reading" §7): a block
// keeps 32 query rows on chip and streams 32-key tiles of K and V, updating
// (m, l, O) per row with the online softmax (§5.2) and normalising once at the
// end.  The backward recomputes P from L (§5.4) in two passes, one owning key
// rows (dK, dV) and one owning query rows (dQ), so nothing needs atomics.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <cfloat>
#include <cmath>
#include <cstdint>

#include "kernels.h"

namespace fa {
namespace {

constexpr int kRows = 32;     // rows per block (4 per warp)
constexpr int kTile = 32;     // keys (or queries) per streamed tile
constexpr int kThreads = 256;
constexpr int kMaxD = 256;
constexpr int kPerLane = kMaxD / 32;

__device__ __forceinline__ float ld(const float* p, int64_t i) { return p[i]; }
__device__ __forceinline__ float ld(const __nv_bfloat16* p, int64_t i) { return __bfloat162float(p[i]); }
__device__ __forceinline__ float ld(const __half* p, int64_t i) { return __half2float(p[i]); }

__device__ __forceinline__ void st(float* p, int64_t i, float v) { p[i] = v; }
__device__ __forceinline__ void st(__nv_bfloat16* p, int64_t i, float v) { p[i] = __float2bfloat16_rn(v); }
__device__ __forceinline__ void st(__half* p, int64_t i, float v) { p[i] = __float2half_rn(v); }

__device__ __forceinline__ float warp_max(float v) {
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Load rows [r0, r0+rows) of a [n][d] matrix into smem (fp32, row stride ld_s), zero past n.
template <typename T>
__device__ __forceinline__ void load_rows(float* s, int ld_s, const T* g, int r0, int rows, int n, int d) {
  for (int i = threadIdx.x; i < rows * d; i += blockDim.x) {
    int r = i / d, c = i - r * d;
    s[r * ld_s + c] = (r0 + r < n) ? ld(g, (int64_t)(r0 + r) * d + c) : 0.f;
  }
}

// ---------------------------------------------------------------------------
// forward
// ---------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(kThreads) fwd_simt(const T* __restrict__ Q, const T* __restrict__ K,
                                                     const T* __restrict__ V, T* __restrict__ O,
                                                     float* __restrict__ L, int n, int d, float scale, int causal,
                                                     int row_tiles, int group, unsigned long long* counter) {
  extern __shared__ float sm[];
  float* qs = sm;                       // [32][d]
  float* ks = qs + kRows * d;           // [32][d+1]
  float* vs = ks + kTile * (d + 1);     // [32][d]
  const int bh = blockIdx.x / row_tiles;
  const int r0 = (blockIdx.x - bh * row_tiles) * kRows;
  const int64_t hoff = (int64_t)bh * n * d;
  const int64_t kvoff = (int64_t)(bh / group) * n * d;  // key/value head of this query head
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int per_lane = (d + 31) / 32;

  load_rows(qs, d, Q + hoff, r0, kRows, n, d);

  float m[4], l[4], acc[4][kPerLane];
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    m[t] = -INFINITY;
    l[t] = 0.f;
#pragma unroll
    for (int i = 0; i < kPerLane; ++i) acc[t][i] = 0.f;
  }
  const int kend = causal ? min(n, r0 + kRows) : n;
  unsigned long long tiles = 0;
  for (int k0 = 0; k0 < kend; k0 += kTile) {
    __syncthreads();
    load_rows(ks, d + 1, K + kvoff, k0, kTile, n, d);
    load_rows(vs, d, V + kvoff, k0, kTile, n, d);
    __syncthreads();
    ++tiles;
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const int rl = warp * 4 + t, row = r0 + rl;
      if (row >= n) continue;  // warp-uniform
      const int key = k0 + lane;
      float s = -INFINITY;
      if (key < n && (!causal || key <= row)) {
        float dot = 0.f;
        for (int c = 0; c < d; ++c) dot = fmaf(qs[rl * d + c], ks[lane * (d + 1) + c], dot);
        s = dot * scale;
      }
      const float mt = warp_max(s);
      const float m_new = fmaxf(m[t], mt);
      if (m_new == -INFINITY) continue;  // nothing visible yet in this row
      const float p = (s == -INFINITY) ? 0.f : expf(s - m_new);
      const float alpha = (m[t] == -INFINITY) ? 0.f : expf(m[t] - m_new);
      l[t] = l[t] * alpha + warp_sum(p);
      m[t] = m_new;
#pragma unroll
      for (int i = 0; i < kPerLane; ++i) acc[t][i] *= alpha;
      for (int j = 0; j < kTile; ++j) {
        const float pj = __shfl_sync(0xffffffffu, p, j);
#pragma unroll
        for (int i = 0; i < kPerLane; ++i) {
          const int c = lane + 32 * i;
          if (i < per_lane && c < d) acc[t][i] = fmaf(pj, vs[j * d + c], acc[t][i]);
        }
      }
    }
  }
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    const int row = r0 + warp * 4 + t;
    if (row >= n) continue;
    const float inv = l[t] > 0.f ? 1.f / l[t] : 0.f;
#pragma unroll
    for (int i = 0; i < kPerLane; ++i) {
      const int c = lane + 32 * i;
      if (i < per_lane && c < d) st(O, hoff + (int64_t)row * d + c, acc[t][i] * inv);
    }
    if (lane == 0) L[(int64_t)bh * n + row] = l[t] > 0.f ? m[t] + logf(l[t]) : -INFINITY;
  }
  if (counter && threadIdx.x == 0) atomicAdd(counter, tiles);
}

// ---------------------------------------------------------------------------
// backward: key-row pass (dK, dV)
// ---------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(kThreads) bwd_dkdv_simt(const T* __restrict__ Q, const T* __restrict__ K,
                                                          const T* __restrict__ V, const T* __restrict__ dO,
                                                          const float* __restrict__ lse2,
                                                          const float* __restrict__ delta, int npad, T* __restrict__ dK,
                                                          T* __restrict__ dV, int n, int d, float scale, int causal,
                                                          int row_tiles, int group) {
  extern __shared__ float sm[];
  float* kb = sm;                        // [32][d] this block's key rows
  float* vb = kb + kRows * d;            // [32][d]
  float* qs = vb + kRows * d;            // [32][d+1] query tile
  float* dos = qs + kTile * (d + 1);     // [32][d+1]
  float* ls = dos + kTile * (d + 1);     // [32]
  float* ds_ = ls + kTile;               // [32]
  const int kvh = blockIdx.x / row_tiles;  // key/value head; its query heads are kvh*group .. +group-1
  const int j0 = (blockIdx.x - kvh * row_tiles) * kRows;
  const int64_t kvoff = (int64_t)kvh * n * d;
  const float scale_log2 = scale * 1.4426950408889634f;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int per_lane = (d + 31) / 32;
  load_rows(kb, d, K + kvoff, j0, kRows, n, d);
  load_rows(vb, d, V + kvoff, j0, kRows, n, d);
  float dk[4][kPerLane], dv[4][kPerLane];
#pragma unroll
  for (int t = 0; t < 4; ++t)
#pragma unroll
    for (int i = 0; i < kPerLane; ++i) dk[t][i] = dv[t][i] = 0.f;
  const int qstart = causal ? (j0 / kTile) * kTile : 0;
  for (int g = 0; g < group; ++g)
  for (int q0 = qstart; q0 < n; q0 += kTile) {
    const int bh = kvh * group + g;  // query head
    const int64_t hoff = (int64_t)bh * n * d;
    __syncthreads();
    load_rows(qs, d + 1, Q + hoff, q0, kTile, n, d);
    load_rows(dos, d + 1, dO + hoff, q0, kTile, n, d);
    if (threadIdx.x < kTile) {
      const int qi = q0 + threadIdx.x;
      ls[threadIdx.x] = qi < n ? lse2[(int64_t)bh * npad + qi] : -INFINITY;
      ds_[threadIdx.x] = qi < n ? delta[(int64_t)bh * npad + qi] : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const int jl = warp * 4 + t, key = j0 + jl;
      if (key >= n) continue;
      const int qi = q0 + lane;
      float p = 0.f, dsv = 0.f;
      if (qi < n && (!causal || qi >= key)) {
        float s = 0.f, dp = 0.f;
        for (int c = 0; c < d; ++c) {
          s = fmaf(qs[lane * (d + 1) + c], kb[jl * d + c], s);
          dp = fmaf(dos[lane * (d + 1) + c], vb[jl * d + c], dp);
        }
        p = exp2f(fmaf(s, scale_log2, ls[lane]));
        dsv = p * (dp - ds_[lane]);
      }
      for (int r = 0; r < kTile; ++r) {
        const float pr = __shfl_sync(0xffffffffu, p, r);
        const float dr = __shfl_sync(0xffffffffu, dsv, r);
#pragma unroll
        for (int i = 0; i < kPerLane; ++i) {
          const int c = lane + 32 * i;
          if (i < per_lane && c < d) {
            dv[t][i] = fmaf(pr, dos[r * (d + 1) + c], dv[t][i]);
            dk[t][i] = fmaf(dr, qs[r * (d + 1) + c], dk[t][i]);
          }
        }
      }
    }
  }
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    const int key = j0 + warp * 4 + t;
    if (key >= n) continue;
#pragma unroll
    for (int i = 0; i < kPerLane; ++i) {
      const int c = lane + 32 * i;
      if (i < per_lane && c < d) {
        st(dK, kvoff + (int64_t)key * d + c, dk[t][i] * scale);
        st(dV, kvoff + (int64_t)key * d + c, dv[t][i]);
      }
    }
  }
}

// ---------------------------------------------------------------------------
// backward: query-row pass (dQ, unscaled, written to the fp32 accumulator)
// ---------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(kThreads) bwd_dq_simt(const T* __restrict__ Q, const T* __restrict__ K,
                                                        const T* __restrict__ V, const T* __restrict__ dO,
                                                        const float* __restrict__ lse2, const float* __restrict__ delta,
                                                        int npad, float* __restrict__ dq_acc, int n, int d,
                                                        float scale, int causal, int row_tiles, int group) {
  extern __shared__ float sm[];
  float* qs = sm;                     // [32][d]
  float* dos = qs + kRows * d;        // [32][d]
  float* ks = dos + kRows * d;        // [32][d+1]
  float* vs = ks + kTile * (d + 1);   // [32][d+1]
  const int bh = blockIdx.x / row_tiles;
  const int r0 = (blockIdx.x - bh * row_tiles) * kRows;
  const int64_t hoff = (int64_t)bh * n * d;
  const int64_t kvoff = (int64_t)(bh / group) * n * d;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int per_lane = (d + 31) / 32;
  const float scale_log2 = scale * 1.4426950408889634f;
  load_rows(qs, d, Q + hoff, r0, kRows, n, d);
  load_rows(dos, d, dO + hoff, r0, kRows, n, d);
  float acc[4][kPerLane], lrow[4], drow[4];
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    const int row = r0 + warp * 4 + t;
    lrow[t] = row < n ? lse2[(int64_t)bh * npad + row] : -INFINITY;
    drow[t] = row < n ? delta[(int64_t)bh * npad + row] : 0.f;
#pragma unroll
    for (int i = 0; i < kPerLane; ++i) acc[t][i] = 0.f;
  }
  const int kend = causal ? min(n, r0 + kRows) : n;
  for (int k0 = 0; k0 < kend; k0 += kTile) {
    __syncthreads();
    load_rows(ks, d + 1, K + kvoff, k0, kTile, n, d);
    load_rows(vs, d + 1, V + kvoff, k0, kTile, n, d);
    __syncthreads();
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const int rl = warp * 4 + t, row = r0 + rl;
      if (row >= n) continue;
      const int key = k0 + lane;
      float dsv = 0.f;
      if (key < n && (!causal || key <= row)) {
        float s = 0.f, dp = 0.f;
        for (int c = 0; c < d; ++c) {
          s = fmaf(qs[rl * d + c], ks[lane * (d + 1) + c], s);
          dp = fmaf(dos[rl * d + c], vs[lane * (d + 1) + c], dp);
        }
        const float p = exp2f(fmaf(s, scale_log2, lrow[t]));
        dsv = p * (dp - drow[t]);
      }
      for (int j = 0; j < kTile; ++j) {
        const float dj = __shfl_sync(0xffffffffu, dsv, j);
#pragma unroll
        for (int i = 0; i < kPerLane; ++i) {
          const int c = lane + 32 * i;
          if (i < per_lane && c < d) acc[t][i] = fmaf(dj, ks[j * (d + 1) + c], acc[t][i]);
        }
      }
    }
  }
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    const int row = r0 + warp * 4 + t;
    if (row >= n) continue;
#pragma unroll
    for (int i = 0; i < kPerLane; ++i) {
      const int c = lane + 32 * i;
      if (i < per_lane && c < d) dq_acc[((int64_t)bh * npad + row) * d + c] = acc[t][i];
    }
  }
}

// ---------------------------------------------------------------------------
// backward preprocess (one warp per padded row) and dQ conversion
// ---------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(256) bwd_pre(const T* __restrict__ O, const T* __restrict__ dO,
                                               const float* __restrict__ lse, float* __restrict__ delta,
                                               float* __restrict__ lse2, float* __restrict__ dq_acc, int n, int npad,
                                               int d, int64_t total_rows, unsigned* __restrict__ sched) {
  if (sched && blockIdx.x == 0 && threadIdx.x < 2) sched[threadIdx.x] = 0u;  // the backward's item queue
  const int64_t gw = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (gw >= total_rows) return;
  const int64_t bh = gw / npad;
  const int row = (int)(gw - bh * npad);
  float acc = 0.f;
  if (row < n) {
    const int64_t off = (bh * n + row) * d;
    for (int c = lane; c < d; c += 32) acc = fmaf(ld(dO, off + c), ld(O, off + c), acc);
    acc = warp_sum(acc);
  }
  if (lane == 0) {
    delta[gw] = row < n ? acc : 0.f;
    // -L log2 e; -inf (P = 0) on padding rows and on rows that saw no key (L = -inf)
    const float lv = row < n ? lse[bh * n + row] : -INFINITY;
    lse2[gw] = lv > -INFINITY ? -lv * 1.4426950408889634f : -INFINITY;
  }
  float* q = dq_acc + gw * d;
  for (int c = lane; c < d; c += 32) q[c] = 0.f;
}

template <typename T>
__global__ void __launch_bounds__(256) dq_convert(const float* __restrict__ dq_acc, T* __restrict__ dQ, int n,
                                                  int npad, int d, float scale, int64_t total) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t rowg = i / d;
    const int c = (int)(i - rowg * d);
    const int64_t bh = rowg / n;
    const int64_t row = rowg - bh * n;
    st(dQ, i, scale * dq_acc[(bh * npad + row) * d + c]);
  }
}

// Vectorised variants for 16-bit inputs with d % 8 == 0: each thread moves 16 bytes of
// input (8 elements); a row of d elements is handled by d / 8 consecutive threads.
template <typename T>
__global__ void __launch_bounds__(256) bwd_pre_vec(const T* __restrict__ O, const T* __restrict__ dO,
                                                   const float* __restrict__ lse, float* __restrict__ delta,
                                                   float* __restrict__ lse2, float* __restrict__ dq_acc, int n,
                                                   int npad, int d, int64_t total_rows, unsigned* __restrict__ sched) {
  if (sched && blockIdx.x == 0 && threadIdx.x < 2) sched[threadIdx.x] = 0u;  // the backward's item queue
  const int tpr = d / 8;  // threads per row: 8, 16 or 32 (power of two)
  const int64_t gt = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t grow = gt / tpr;
  const int sub = (int)(gt - grow * tpr);
  const bool active = grow < total_rows;
  const int64_t bh = active ? grow / npad : 0;
  const int row = active ? (int)(grow - bh * npad) : 0;
  float acc = 0.f;
  if (active && row < n) {
    const int64_t off = (bh * n + row) * d + sub * 8;
    const uint4 a = *reinterpret_cast<const uint4*>(O + off);
    const uint4 b = *reinterpret_cast<const uint4*>(dO + off);
    const T* pa = reinterpret_cast<const T*>(&a);
    const T* pb = reinterpret_cast<const T*>(&b);
#pragma unroll
    for (int i = 0; i < 8; ++i) acc = fmaf(ld(pa, i), ld(pb, i), acc);
  }
  for (int o = tpr >> 1; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if (!active) return;
  if (sub == 0) {
    delta[grow] = row < n ? acc : 0.f;
    const float lv = row < n ? lse[bh * n + row] : -INFINITY;
    lse2[grow] = lv > -INFINITY ? -lv * 1.4426950408889634f : -INFINITY;
  }
  float4* q = reinterpret_cast<float4*>(dq_acc + grow * d + sub * 8);
  q[0] = make_float4(0.f, 0.f, 0.f, 0.f);
  q[1] = make_float4(0.f, 0.f, 0.f, 0.f);
}

template <typename T>
__global__ void __launch_bounds__(256) dq_convert_vec(const float* __restrict__ dq_acc, T* __restrict__ dQ, int n,
                                                      int npad, int d, float scale, int64_t total8) {
  for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < total8;
       t += (int64_t)gridDim.x * blockDim.x) {
    const int64_t e = t * 8;
    const int64_t rowg = e / d;
    const int c = (int)(e - rowg * d);
    const int64_t bh = rowg / n;
    const int64_t src = (bh * npad + (rowg - bh * n)) * d + c;
    const float4 x0 = *reinterpret_cast<const float4*>(dq_acc + src);
    const float4 x1 = *reinterpret_cast<const float4*>(dq_acc + src + 4);
    uint4 out;
    T* po = reinterpret_cast<T*>(&out);
    st(po, 0, scale * x0.x); st(po, 1, scale * x0.y); st(po, 2, scale * x0.z); st(po, 3, scale * x0.w);
    st(po, 4, scale * x1.x); st(po, 5, scale * x1.y); st(po, 6, scale * x1.z); st(po, 7, scale * x1.w);
    *reinterpret_cast<uint4*>(dQ + e) = out;
  }
}

template <typename F, typename... Args>
cudaError_t launch_smem(F kern, int grid, size_t smem, cudaStream_t s, Args... args) {
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  kern<<<grid, kThreads, smem, s>>>(args...);
  return cudaGetLastError();
}

template <typename T>
cudaError_t fwd_simt_t(const FwdArgs& a) {
  const int tiles = (a.n + kRows - 1) / kRows;
  const size_t smem = sizeof(float) * (size_t)(kRows * a.d + kTile * (a.d + 1) + kTile * a.d);
  return launch_smem(fwd_simt<T>, a.bh * tiles, smem, a.stream, (const T*)a.q, (const T*)a.k, (const T*)a.v,
                     (T*)a.o, a.lse, a.n, a.d, a.scale, a.causal, tiles, a.group, a.counter);
}

template <typename T>
cudaError_t bwd_simt_t(const BwdArgs& a) {
  const int tiles = (a.n + kRows - 1) / kRows;
  const int npad = (int)padded_rows(a.n);
  const size_t smem1 = sizeof(float) * (size_t)(2 * kRows * a.d + 2 * kTile * (a.d + 1) + 2 * kTile);
  cudaError_t e = launch_smem(bwd_dkdv_simt<T>, (a.bh / a.group) * tiles, smem1, a.stream, (const T*)a.q, (const T*)a.k,
                              (const T*)a.v, (const T*)a.dout, (const float*)a.lse2, (const float*)a.delta, npad,
                              (T*)a.dk, (T*)a.dv, a.n, a.d, a.scale, a.causal, tiles, a.group);
  if (e != cudaSuccess) return e;
  const size_t smem2 = sizeof(float) * (size_t)(2 * kRows * a.d + 2 * kTile * (a.d + 1));
  return launch_smem(bwd_dq_simt<T>, a.bh * tiles, smem2, a.stream, (const T*)a.q, (const T*)a.k, (const T*)a.v,
                     (const T*)a.dout, (const float*)a.lse2, (const float*)a.delta, npad, a.dq_acc, a.n, a.d,
                     a.scale, a.causal, tiles, a.group);
}

template <typename T>
cudaError_t pre_t(const BwdArgs& a) {
  const int npad = (int)padded_rows(a.n);
  const int64_t rows = (int64_t)a.bh * npad;
  if (sizeof(T) == 2 && (a.d == 64 || a.d == 128 || a.d == 256)) {
    const int64_t threads = rows * (a.d / 8);
    bwd_pre_vec<T><<<(unsigned)((threads + 255) / 256), 256, 0, a.stream>>>(
        (const T*)a.o, (const T*)a.dout, a.lse, a.delta, a.lse2, a.dq_acc, a.n, npad, a.d, rows, a.sched);
    return cudaGetLastError();
  }
  const int64_t blocks = (rows * 32 + 255) / 256;
  bwd_pre<T><<<(unsigned)blocks, 256, 0, a.stream>>>((const T*)a.o, (const T*)a.dout, a.lse, a.delta, a.lse2,
                                                     a.dq_acc, a.n, npad, a.d, rows, a.sched);
  return cudaGetLastError();
}

template <typename T>
cudaError_t convert_t(const BwdArgs& a) {
  const int npad = (int)padded_rows(a.n);
  const int64_t total = (int64_t)a.bh * a.n * a.d;
  if (sizeof(T) == 2 && a.d % 8 == 0) {
    const int64_t total8 = total / 8;
    int64_t blocks = (total8 + 255) / 256;
    if (blocks > 152 * 16) blocks = 152 * 16;
    dq_convert_vec<T><<<(unsigned)blocks, 256, 0, a.stream>>>(a.dq_acc, (T*)a.dq, a.n, npad, a.d, a.scale, total8);
    return cudaGetLastError();
  }
  int64_t blocks = (total + 255) / 256;
  if (blocks > 152 * 64) blocks = 152 * 64;
  dq_convert<T><<<(unsigned)blocks, 256, 0, a.stream>>>(a.dq_acc, (T*)a.dq, a.n, npad, a.d, a.scale, total);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_simt(const FwdArgs& a) {
  switch (a.dtype) {
    case DT_BF16: return fwd_simt_t<__nv_bfloat16>(a);
    case DT_FP16: return fwd_simt_t<__half>(a);
    default: return fwd_simt_t<float>(a);
  }
}

cudaError_t launch_bwd_simt(const BwdArgs& a) {
  switch (a.dtype) {
    case DT_BF16: return bwd_simt_t<__nv_bfloat16>(a);
    case DT_FP16: return bwd_simt_t<__half>(a);
    default: return bwd_simt_t<float>(a);
  }
}

cudaError_t launch_bwd_pre(const BwdArgs& a) {
  switch (a.dtype) {
    case DT_BF16: return pre_t<__nv_bfloat16>(a);
    case DT_FP16: return pre_t<__half>(a);
    default: return pre_t<float>(a);
  }
}

cudaError_t launch_dq_convert(const BwdArgs& a) {
  switch (a.dtype) {
    case DT_BF16: return convert_t<__nv_bfloat16>(a);
    case DT_FP16: return convert_t<__half>(a);
    default: return convert_t<float>(a);
  }
}

}  // namespace fa
