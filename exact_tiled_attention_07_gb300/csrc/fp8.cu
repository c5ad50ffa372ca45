// FP8 (E4M3) path: block quantisation, and the tensor-core forward on quantised Q, K, V.
//
// "Lecture 8 · GPU Performance & FlashAttention" §8.1 and "FlashAttention and GPU memory" §11:
// the third generation runs attention in 8-bit floating point with block quantisation, one
// scale per block of each tensor.  Here a block is 128 rows x d of one head (the tile the
// kernel streams), its scale is amax / 448 (E4M3's largest finite value) and its codes are
// E4M3(x / scale), rounded to nearest even; the scale and the quotient are fp32 divisions.
//
// fwd_fp8_kernel is the 16-bit forward's pipeline (two query tiles ping-ponging, TMA ring,
// softmax in the exp2 domain with lazy rescaling) with 8-bit operands: S = Q8 K8^T and
// O += P8 V8 are kind::f8f6f4 MMAs (K = 32 per instruction).  The block scales enter as
//   S_ij = tau * sq(i) * sk(j) * (Q8 K8^T)_ij        (one factor per pair of tiles),
//   O_i  = sum_j P_ij sv(j) V8_j / l_i,
// with sv(j) folded into P before it is rounded to E4M3: P8 = E4M3(exp2(S st + log2 sv(j) - m)),
// where the online softmax's running maximum m is taken over S st + log2 sv(j): so P8 <= 2^8
// (the lazy-rescale bound) stays inside E4M3's range and a row's largest V-weighted
// probabilities stay near 1 whatever the spread of the V scales (a head-wide reference, the
// head's largest V scale, let the probabilities of small-scale blocks sink into E4M3's subnormal
// range).  l sums the unrounded probabilities exp2(S st - m) (each tile's sum divided by sv(j)),
// and the epilogue divides O by l.
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

// ------------------------------------------------------------------------------ forward

constexpr int BM = 128;  // query rows per tile
constexpr int BN = 128;  // keys per tile
constexpr float kRescaleThreshold = 8.0f;

// d = 128: one 128-byte row per tile row (128-byte swizzle); d = 64: one 64-byte row (64-byte
// swizzle); either way every tile is a single TMA box
template <int D_>
struct Fp8Cfg {
  static constexpr int D = D_;
  static constexpr int SW = D;                // swizzle width in bytes = row length
  static constexpr int NQ = 2;
  static constexpr int TILE_BYTES = 128 * D;  // 16 / 8 KB (Q, K or V tile)
  static constexpr int STAGES = D == 128 ? 12 : 24;
  static constexpr int PRODUCER_WARP = 8;
  static constexpr int MMA_WARP = 9;
  static constexpr int THREADS = 320;
  static constexpr int S_COL0 = 0, S_COL1 = 128, O_COL0 = 256, O_COL1 = 256 + D;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_RING = NQ * TILE_BYTES;
  static constexpr int OFF_BAR = OFF_RING + STAGES * TILE_BYTES;
  // q_full, kv_full/empty ring, s/p/o_full [2] each, drain, o_empty [2], q_empty, item_full/empty [2]
  static constexpr int NBAR = 1 + 2 * STAGES + 2 + 2 + 2 + 1 + 2 + 1 + 4;
  static constexpr int OFF_RED = OFF_BAR + NBAR * 8 + 32;  // [2][8] floats: per-warp partial maxima
  static constexpr int SMEM = OFF_RED + 16 * 4;
};

// Persistent like the 16-bit forward: a CTA per SM walks work items (head, two query tiles),
// from the queue when the launch has a slot (QUEUE) or in grid order; q_empty lets an item's Q
// load once the last S of the previous item is issued, o_empty lets an item's first P V overwrite
// O once the softmax has read it, and every phase runs on counters that continue across items.
template <int DH, bool OUT_BF16, bool QUEUE>
__global__ void __launch_bounds__(Fp8Cfg<DH>::THREADS, 1)
    fwd_fp8_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const float* __restrict__ q_scales,
                   const float* __restrict__ k_scales, const float* __restrict__ v_scales, void* __restrict__ out,
                   float* __restrict__ lse, int n, int bh_count, int tiles_per_head, float scale_log2, int causal,
                   int group, unsigned long long* err, unsigned long long* counter, unsigned* __restrict__ sched,
                   int hgroup) {
  using C = Fp8Cfg<DH>;
  constexpr int D = C::D;
  extern __shared__ __align__(1024) uint8_t smem[];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* q_full = bars;
  uint64_t* kv_full = bars + 1;
  uint64_t* kv_empty = bars + 1 + C::STAGES;
  uint64_t* s_full = bars + 1 + 2 * C::STAGES;  // [2]
  uint64_t* p_full = s_full + 2;                // [2]
  uint64_t* o_full = p_full + 2;                // [2]
  uint64_t* drain = o_full + 2;
  uint64_t* o_empty = drain + 1;                // [2] the softmax has read O_q of its last item
  uint64_t* q_empty = o_empty + 2;              // every S of the last item is issued and done
  uint64_t* item_full = q_empty + 1;            // [2] (queue mode)
  uint64_t* item_empty = item_full + 2;         // [2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::NBAR);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* item_slot = reinterpret_cast<volatile int*>(tmem_slot + 2);  // [2]
  const ErrCtx ctx{err, abort_flag};

  const int nblk = (n + BN - 1) / BN;  // 128-row blocks per head: key tiles and scale entries
  const int total_items = bh_count * tiles_per_head;
  struct Item {
    int head, kvhead, qrow0;
    int nq[2];  // key tiles of each query tile
  };
  // work items: head-major (CTAs running together share K/V in L2); causal: heaviest (last)
  // query tiles first within groups of heads
  auto item_of = [&](int item) {
    Item w;
    int tile;
    if (causal) {
      int rank;
      grouped_work_item(item, bh_count, tiles_per_head, hgroup, &w.head, &rank);
      tile = tiles_per_head - 1 - rank;
    } else {
      w.head = item / tiles_per_head;
      tile = item - w.head * tiles_per_head;
    }
    w.kvhead = w.head / group;
    w.qrow0 = tile * (C::NQ * BM);
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const int first = w.qrow0 + q * BM;
      if (first >= n) {
        w.nq[q] = 0;
      } else if (causal) {
        w.nq[q] = min(nblk, (min(first + BM, n) - 1) / BN + 1);
      } else {
        w.nq[q] = nblk;
      }
    }
    return w;
  };
  // the static order: rounds of gridDim.x items (the grid size and CTA index read afresh each time)
  auto nth_item = [&](int r) {
    const int64_t item = (int64_t)r * (int)grid_dim_x() + (int)cta_id_x();
    return item < total_items ? (int)item : -1;
  };
  // a consumer warp's r-th item: queue mode reads the producer's slot r % 2 (every consumer warp
  // reads every slot once; `good` turns false, and the item -1, when the bounded wait ran out)
  auto next_item = [&](int r, bool& good) {
    if constexpr (!QUEUE) return nth_item(r);
    const int t = r & 1;
    good = __all_sync(0xffffffffu, mbar_wait(item_full + t, (uint32_t)(r >> 1) & 1, ctx, 250)) && good;
    const int item = good ? item_slot[t] : -1;
    __syncwarp();
    if (lane == 0) mbar_arrive(item_empty + t);
    return item;
  };

  if (threadIdx.x == 0) {
    if ((smem_u32(smem) & 1023u) != 0) report_error(err, DERR_BAD_SMEM_ALIGN, 0);
    *abort_flag = (smem_u32(smem) & 1023u) != 0;
    mbar_init(q_full, 1);
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(kv_full + s, 1);
      mbar_init(kv_empty + s, 1);
    }
    for (int q = 0; q < 2; ++q) {
      mbar_init(s_full + q, 1);
      mbar_init(p_full + q, 128);
      mbar_init(o_full + q, 1);
      mbar_init(o_empty + q, 128);
      mbar_init(item_full + q, 1);
      mbar_init(item_empty + q, 9);  // the eight softmax warps and the MMA warp
    }
    mbar_init(drain, 1);
    mbar_init(q_empty, 1);
    fence_barrier_init();
  }
  if (warp == C::MMA_WARP) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  const bool start_ok = (*abort_flag == 0);

  if (warp == C::PRODUCER_WARP) {
    // ------------------------------------------------------------------ TMA producer
    if (start_ok && lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      uint32_t ring_pos = 0;  // ring loads issued (all items)
      int q_loads = 0;
      bool ok = true;
      // the r-th item: queue mode draws a ticket and publishes the item, or -1 once the queue is
      // empty, when every reader of the slot's previous item has it
      auto draw = [&](int r) {
        if constexpr (!QUEUE) return nth_item(r);
        if (r >= 2 && !(ok = mbar_wait(item_empty + (r & 1), (uint32_t)((r - 2) >> 1) & 1, ctx, 214))) return -1;
        const unsigned ticket = atomicAdd(sched, 1u);
        const int item = ticket < (unsigned)total_items ? (int)ticket : -1;
        item_slot[r & 1] = item;
        mbar_arrive(item_full + (r & 1));
        return item;
      };
      for (int r = 0, item = draw(0); ok && item >= 0; item = draw(++r)) {
        const Item w = item_of(item);
        const int nmax = max(w.nq[0], w.nq[1]);
        // Q of this item once the previous item's S = Q K^T are done
        if (q_loads > 0 && !(ok = mbar_wait(q_empty, (q_loads - 1) & 1, ctx, 213))) break;
        mbar_arrive_expect_tx(q_full, C::NQ * C::TILE_BYTES);
        for (int q = 0; q < C::NQ; ++q)
          tma_load_3d(smem + C::OFF_Q + q * C::TILE_BYTES, &tm_q, q_full, 0, w.qrow0 + q * BM, w.head);
        ++q_loads;
        for (int idx = 0; idx < 2 * nmax; ++idx) {
          const uint32_t g = ring_pos;
          const int slot = g % C::STAGES, use = g / C::STAGES;
          if (use > 0 && !(ok = mbar_wait(kv_empty + slot, (use - 1) & 1, ctx, 210))) break;
          mbar_arrive_expect_tx(kv_full + slot, C::TILE_BYTES);
          tma_load_3d(smem + C::OFF_RING + slot * C::TILE_BYTES, (idx & 1) ? &tm_v : &tm_k, kv_full + slot, 0,
                      (idx >> 1) * BN, w.kvhead);
          ++ring_pos;
        }
      }
      // drain: every copy this thread started must land before the CTA may exit
      ErrCtx nctx = ctx;
      int no_abort = 0;
      nctx.abort = &no_abort;
      if (q_loads > 0) mbar_wait(q_full, (q_loads - 1) & 1, nctx, 211);
      for (int g = (int)ring_pos - 1; g >= 0 && g >= (int)ring_pos - C::STAGES; --g)
        mbar_wait(kv_full + g % C::STAGES, (g / C::STAGES) & 1, nctx, 212);
    }
    __syncwarp();
  } else if (warp == C::MMA_WARP) {
    // ------------------------------------------------------------------ MMA issuer
    if (start_ok) {
      const bool leader = elect_one_sync();
      // E4M3 is format code 0 in the A/B fields: the f16 descriptor layout with the f16 codes
      const uint32_t idesc_qk = make_idesc_f16(BM, BN, false, false, false);
      const uint32_t idesc_pv = make_idesc_f16(BM, D, false, false, true);
      const uint32_t q_base = smem_u32(smem + C::OFF_Q);
      const uint32_t ring = smem_u32(smem + C::OFF_RING);
      uint32_t ring_pos = 0;  // ring entry of the item's first K tile (all items so far)
      int tq[2] = {0, 0};     // key tiles processed by each query tile (all items): P phases
      int oq[2] = {0, 0};     // items with a result for each query tile: O phases
      int items = 0;
      auto slot_of = [&](int idx) { return (int)((ring_pos + idx) % C::STAGES); };
      auto wait = [&](uint64_t* b, uint32_t parity, uint32_t site) {
        return __all_sync(0xffffffffu, mbar_wait(b, parity, ctx, site));
      };
      auto wait_full = [&](int idx) {
        return wait(kv_full + slot_of(idx), ((ring_pos + idx) / C::STAGES) & 1, 220);
      };
      auto commit = [&](uint64_t* b) {
        if (leader) umma_commit(b);
        __syncwarp();
      };
      // K-major 8-bit tile rows of D bytes in 8-row swizzle atoms of 8 D bytes
      auto sdesc = [](uint32_t addr, uint32_t lbo, uint32_t sbo) {
        return C::SW == 128 ? make_sdesc_sw128(addr, lbo, sbo) : make_sdesc_sw64(addr, lbo, sbo);
      };
      // S = Q8_q K8^T: 32 bytes (32 elements) of the D-byte rows per instruction
      auto issue_qk = [&](int q, int kidx, uint32_t s_col) {
        const uint32_t kt = ring + slot_of(kidx) * C::TILE_BYTES;
        const uint32_t qt = q_base + q * C::TILE_BYTES;
        uint64_t ad[D / 32], bd[D / 32];
#pragma unroll
        for (int kk = 0; kk < D / 32; ++kk) {
          ad[kk] = sdesc(qt + kk * 32, 16, 8 * C::SW);
          bd[kk] = sdesc(kt + kk * 32, 16, 8 * C::SW);
        }
        if (leader) {
#pragma unroll
          for (int kk = 0; kk < D / 32; ++kk) umma_ss_f8(tbase + s_col, ad[kk], bd[kk], idesc_qk, kk > 0);
        }
        __syncwarp();
      };
      // O += P8 V8: P8 (4 keys per TMEM column) in [p_col, p_col + 32); V8 MN-major (the d bytes
      // of a key contiguous), 32 keys (4 swizzle atoms of 8 rows) per instruction
      auto issue_pv = [&](uint32_t o_col, uint32_t p_col, int vidx, bool acc) {
        const uint32_t vt = ring + slot_of(vidx) * C::TILE_BYTES;
        uint64_t bd[BN / 32];
#pragma unroll
        for (int kk = 0; kk < BN / 32; ++kk) bd[kk] = sdesc(vt + kk * 32 * C::SW, BN * C::SW, 8 * C::SW);
        if (leader) {
#pragma unroll
          for (int kk = 0; kk < BN / 32; ++kk)
            umma_ts_f8(tbase + o_col, tbase + p_col + kk * 8, bd[kk], idesc_pv, (acc || kk > 0) ? 1u : 0u);
        }
        __syncwarp();
      };
      // the first P V of query tile q in an item overwrites O_q: the softmax must have read it
      auto o_free = [&](int q) { return oq[q] == 0 || wait(o_empty + q, (oq[q] - 1) & 1, 226 + q); };
      bool ok = true;
      for (int r = 0, item = next_item(0, ok); ok && item >= 0; item = next_item(++r, ok)) {
        const Item w = item_of(item);
        const int* nq = w.nq;
        const int nmax = max(nq[0], nq[1]);
        if (!(ok = wait(q_full, items & 1, 221))) break;
        tc_fence_after();
        if (nmax > 0) {
          if (!(ok = wait_full(0))) break;
          tc_fence_after();
          if (nq[0] > 0) { issue_qk(0, 0, C::S_COL0); commit(s_full + 0); }
          if (nq[1] > 0) { issue_qk(1, 0, C::S_COL1); commit(s_full + 1); }
          commit(kv_empty + slot_of(0));
        }
        if (nmax <= 1) commit(q_empty);  // every S of the item is issued
        for (int j = 0; ok && j < nmax; ++j) {
          const int vidx = 2 * j + 1, kidx = 2 * j + 2;
          if (!(ok = wait_full(vidx))) break;
          if (j < nq[0]) {
            if (!(ok = wait(p_full + 0, (tq[0] + j) & 1, 222))) break;
            if (j == 0 && !(ok = o_free(0))) break;
            tc_fence_after();
            issue_pv(C::O_COL0, C::S_COL0, vidx, j > 0);
          }
          if (j + 1 < nmax) {
            if (!(ok = wait_full(kidx))) break;
            tc_fence_after();
          }
          if (j + 1 < nq[0]) { issue_qk(0, kidx, C::S_COL0); commit(s_full + 0); }
          if (j < nq[1]) {
            if (!(ok = wait(p_full + 1, (tq[1] + j) & 1, 223))) break;
            if (j == 0 && !(ok = o_free(1))) break;
            tc_fence_after();
            issue_pv(C::O_COL1, C::S_COL1, vidx, j > 0);
          }
          commit(kv_empty + slot_of(vidx));
          if (j + 1 < nq[1]) { issue_qk(1, kidx, C::S_COL1); commit(s_full + 1); }
          if (j + 1 < nmax) commit(kv_empty + slot_of(kidx));
          if (j == nmax - 2) commit(q_empty);  // the item's last S are issued
          if (j == nq[0] - 1) commit(o_full + 0);
          if (j == nq[1] - 1) commit(o_full + 1);
        }
        ring_pos += 2 * nmax;
        for (int q = 0; q < 2; ++q) {
          tq[q] += nq[q];
          oq[q] += nq[q] > 0 ? 1 : 0;
        }
        ++items;
      }
      ErrCtx nctx = ctx;
      int no_abort = 0;
      nctx.abort = &no_abort;
      commit(drain);
      mbar_wait(drain, 0, nctx, 225);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------ softmax warpgroups
    const int q = warp >> 2;
    const int quarter = warp & 3;
    const uint32_t lane_base = quarter * 32;
    const int rit = quarter * 32 + lane;
    const uint32_t s_col = q ? C::S_COL1 : C::S_COL0;
    const uint32_t o_col = q ? C::O_COL1 : C::O_COL0;
    int tq = 0;  // key tiles this query tile processed (all items): S / P phases
    int oq = 0;  // items with a result: O phases
    bool ok = start_ok;
    // The eight softmax warps meet at a named barrier per item and decide together, through that
    // barrier's reduction, whether to take another item: a warp whose bounded wait ran out cannot
    // leave the others waiting there.
    for (int r = 0;; ++r) {
      bool got = ok;
      const int item = next_item(r, got);
      const bool have = got && item >= 0;
      const Item w = item_of(have ? item : 0);
      if (!named_bar_and(1, 256, have)) break;
      const float* vs = v_scales + (int64_t)w.kvhead * nblk;
      const int head = w.head;
      const int row = w.qrow0 + q * BM + rit;
      const int nb = w.nq[q];
      const float* ks = k_scales + (int64_t)w.kvhead * nblk;
      const int qblk = min((w.qrow0 + q * BM) / BM, nblk - 1);
      const float sq_log2 = scale_log2 * q_scales[(int64_t)head * nblk + qblk];
      float m = -INFINITY;
      float l = 0.f;
      float sk_next = nb > 0 ? ks[0] : 0.f, sv_next = nb > 0 ? vs[0] : 0.f;
      for (int j = 0; ok && j < nb; ++j) {
        const int t = tq + j;
        const float st = sq_log2 * sk_next;  // tau log2(e) sq sk: S units -> log2 units
        const float pv = sv_next;            // the key block's V scale, folded into P's exponent
        const float lpv = __log2f(pv);
        if (j + 1 < nb) {
          sk_next = ks[j + 1];
          sv_next = vs[j + 1];
        }
        ok = __all_sync(0xffffffffu, mbar_wait(s_full + q, t & 1, ctx, 230 + q));
        if (!ok) break;
        tc_fence_after();
        uint32_t sr[BN / 32][32];
#pragma unroll
        for (int c = 0; c < BN / 32; ++c) tmem_ld32(tmem_addr(tbase, lane_base, s_col + c * 32), sr[c]);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < BN / 32; ++c) reg_fence(sr[c]);
        float s[BN];
#pragma unroll
        for (int c = 0; c < BN / 32; ++c)
#pragma unroll
          for (int i = 0; i < 32; ++i) s[c * 32 + i] = __uint_as_float(sr[c][i]);
        int limit = n - j * BN;
        if (causal) limit = min(limit, row - j * BN + 1);
        if (limit < BN) {
#pragma unroll
          for (int c = 0; c < BN; ++c)
            if (c >= limit) s[c] = -INFINITY;
        }
        // the running maximum is over S st + log2 sv: a row's largest V-weighted probability stays
        // near 1 in E4M3, whatever the spread of the V block scales
        const float mx = row_max3(s);
        const float m_blk = mx * st + lpv;
        float alpha = 1.f;
        bool rescale = false;
        if (m == -INFINITY) {
          m = m_blk;
          alpha = 0.f;
        } else if (m_blk > m + kRescaleThreshold) {
          alpha = ex2(m - m_blk);
          m = m_blk;
          rescale = true;
        }
        // P sv = exp2(S st + log2 sv - m): the V factor rides in the exponent, and the row sum of P
        // is that of the scaled values divided by the factor once per tile
        const float neg_m = ((m == -INFINITY) ? 0.f : -m) + lpv;
        // two partial sums of pairs (paired fp32 FMA and adds): no single long add chain
        float2 part[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
        uint32_t pk[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float2 x01 = ffma2(make_float2(s[4 * i], s[4 * i + 1]), st, neg_m);
          const float2 x23 = ffma2(make_float2(s[4 * i + 2], s[4 * i + 3]), st, neg_m);
          const float2 p01 = make_float2(ex2(x01.x), ex2(x01.y)), p23 = make_float2(ex2(x23.x), ex2(x23.y));
          part[i & 1] = fadd2(part[i & 1], fadd2(p01, p23));
          pk[i] = pack4_e4m3(p01.x, p01.y, p23.x, p23.y);
        }
        const float sum = ((part[0].x + part[1].x) + (part[0].y + part[1].y)) / pv;
        tmem_st32(tmem_addr(tbase, lane_base, s_col), pk);
        l = l * alpha + sum;
        if (__any_sync(0xffffffffu, rescale)) {
          // O row *= alpha; O is stable: the PV of block j-1 completed before S_j (same issuing
          // thread, in order)
          const float a = rescale ? alpha : 1.f;
#pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            uint32_t rr[32];
            const uint32_t ta = tmem_addr(tbase, lane_base, o_col + c * 32);
            tmem_ld32(ta, rr);
            tmem_wait_ld();
            reg_fence(rr);
#pragma unroll
            for (int i = 0; i < 32; ++i) rr[i] = __float_as_uint(__uint_as_float(rr[i]) * a);
            tmem_st32(ta, rr);
          }
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(p_full + q);
      }
      // epilogue: O / l -> global (16-bit), L = (m + log2 l) ln 2 (l sums exp2(S st - m), so
      // m + log2 l is the log2-sum-exp of S st whatever V factors m took in)
      if (ok && nb > 0) {
        ok = __all_sync(0xffffffffu, mbar_wait(o_full + q, oq & 1, ctx, 240 + q));
        if (ok) {
          tc_fence_after();
          const float inv = l > 0.f ? 1.f / l : 0.f;
          uint8_t* orow = reinterpret_cast<uint8_t*>(out) + (((int64_t)head * n + row) * D) * 2;
#pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            uint32_t rr[32];
            tmem_ld32(tmem_addr(tbase, lane_base, o_col + c * 32), rr);
            tmem_wait_ld();
            reg_fence(rr);
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
              pk[i] = pack2<OUT_BF16>(__uint_as_float(rr[2 * i]) * inv, __uint_as_float(rr[2 * i + 1]) * inv);
            if (row < n) {
              uint4* dst = reinterpret_cast<uint4*>(orow + c * 64);
#pragma unroll
              for (int i = 0; i < 4; ++i) dst[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
            }
          }
          // every TMEM load of O is done: the next item may overwrite it
          tc_fence_before();
          mbar_arrive(o_empty + q);
          ++oq;
          if (row < n) lse[(int64_t)head * n + row] = l > 0.f ? (m + log2f(l)) * 0.6931471805599453f : -INFINITY;
          if (counter && rit == 0) atomicAdd(counter, (unsigned long long)nb);
        }
      }
      tq += nb;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == C::MMA_WARP) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
  if (QUEUE && threadIdx.x == 0) {
    // this CTA draws no more tickets; the last one to get here empties the queue for the next
    // launch that uses it (every CTA has drawn its last ticket by then)
    __threadfence();
    if (atomicAdd(sched + 1, 1u) == gridDim.x - 1) {
      atomicExch(sched, 0u);
      atomicExch(sched + 1, 0u);
    }
  }
}

template <int DH, bool OUT_BF16>
cudaError_t launch_fwd_fp8_t(const Fp8FwdArgs& a) {
  using C = Fp8Cfg<DH>;
  CUtensorMap tq, tk, tv;
  const int bh_kv = a.bh / a.group;
  if (!make_tmap_8bit_3d(&tq, a.q8, C::D, a.n, a.bh, BM, C::SW) ||
      !make_tmap_8bit_3d(&tk, a.k8, C::D, a.n, bh_kv, BN, C::SW) ||
      !make_tmap_8bit_3d(&tv, a.v8, C::D, a.n, bh_kv, BN, C::SW))
    return cudaErrorInvalidValue;
  const int tiles = (a.n + C::NQ * BM - 1) / (C::NQ * BM);
  const int64_t items = (int64_t)a.bh * tiles;
  const int64_t grid = std::min<int64_t>(items, device_sm_count());
  QueueSlot qs;
  if (grid < items) qs = queue_slot_take(a.stream);
  auto kern = qs.slot >= 0 ? fwd_fp8_kernel<DH, OUT_BF16, true> : fwd_fp8_kernel<DH, OUT_BF16, false>;
  // causal order: groups of query heads whose 8-bit K, V stay in L2
  const int hgroup = head_group_for_l2((int64_t)2 * a.n * C::D / a.group);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e == cudaSuccess) {
    kern<<<(unsigned)grid, C::THREADS, C::SMEM, a.stream>>>(tq, tk, tv, a.q_scales, a.k_scales, a.v_scales, a.o,
                                                            a.lse, a.n, a.bh, tiles, a.scale * 1.4426950408889634f,
                                                            a.causal, a.group, a.err, a.counter, qs.counters, hgroup);
    e = cudaGetLastError();
  }
  return queue_slot_done(qs, e, a.stream);
}

}  // namespace

cudaError_t launch_quantize_fp8(const QuantArgs& a) {
  switch (a.dtype) {
    case DT_BF16: return launch_quantize_t<__nv_bfloat16>(a);
    case DT_FP16: return launch_quantize_t<__half>(a);
    default: return launch_quantize_t<float>(a);
  }
}

bool fwd_fp8_supported(int d) { return d == 64 || d == 128; }

cudaError_t launch_fwd_fp8(const Fp8FwdArgs& a) {
  const bool bf = a.out_dtype == DT_BF16;
  switch (a.d) {
    case 64: return bf ? launch_fwd_fp8_t<64, true>(a) : launch_fwd_fp8_t<64, false>(a);
    case 128: return bf ? launch_fwd_fp8_t<128, true>(a) : launch_fwd_fp8_t<128, false>(a);
    default: return cudaErrorNotSupported;
  }
}

}  // namespace fa
