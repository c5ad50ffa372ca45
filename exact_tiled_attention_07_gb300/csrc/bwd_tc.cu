// Tensor-core backward for bf16/fp16, head dims 64/128/256 (sm_103a: TMA, tcgen05, TMEM).
//
// Recomputing backward ("Lecture 8 · GPU Performance & FlashAttention" §5.4; "FlashAttention
// and GPU memory" §09): nothing N x N was stored, so every (key tile j, query tile i) pair
// recomputes its scores from Q, K and the saved row statistic L:
//     S^T = K_j Q_i^T,   P^T = exp2(S^T tau log2e - L_i log2e)       (= e^(S - m)/l)
// (the workspace holds -L_i log2e, so the exponent is one fused multiply-add)
//     dV_j += P^T dO_i,   dP^T = V_j dO_i^T,   dS^T = P^T o (dP^T - D_i)
//     dK_j += dS^T Q_i,   dQ_i += dS K_j      (tau applied to dK here and to dQ on conversion)
// with D_i = sum_k dO_ik O_ik precomputed by the preprocess kernel (the §5.4 identity).
//
// A work item is a 128-key tile of one key/value head (with grouped-query attention it visits
// every query head of that key/value head): while a CTA works on it, K_j, V_j stay in shared
// memory and the dK_j, dV_j accumulators stay in TMEM, and query tiles (Q_i, dO_i, L_i, D_i)
// stream through a three-stage TMA ring.  The grid is persistent (one CTA per SM, items from a
// queue; see the kernel).  Working transposed puts keys on TMEM lanes, so
// one thread owns one key row: P^T and dS^T need no cross-thread reduction.  K_j, P^T and
// dS^T sit in TMEM as A operands (S^T = K Q^T, dV += P^T dO, dK += dS^T Q), which spares
// the shared-memory read of A that an all-smem MMA pays; dS^T also goes to shared memory
// as an operand of the dQ GEMM.
//
// Roles: two compute warpgroups for the elementwise work (P^T, dS^T), one drain warpgroup, a
// TMA producer warp and an MMA warp.  Both compute warpgroups own the tile's 128 key rows (a
// warp reads the TMEM lanes of its quarter, so warps w and w + 4 see the same rows) and each
// takes half of every step's queries.  dQ
// partials are summed over key tiles in an fp32 accumulator in global memory: the drain
// warpgroup moves each step's dQ partial from TMEM into a shared-memory staging tile as soon as
// it completes, and one thread adds the tile to global memory with a TMA bulk reduction (whole
// 128-byte lines, no per-element atomics); at the end of an item it also stores dK, dV.  Two
// shapes of the dQ GEMM keep every TMEM region separate, so no GEMM waits for another region to
// be drained:
//   d = 64:  128 queries per step, dQ = dS K   (M = 128 queries, N = 64)
//   d = 128:  64 queries per step, dQ^T = K^T dS^T (M = 128 = d, N = 64 queries)
//   d = 256:  32 queries per step, one half of d per work item: dQ^T of that half
//             (M = 128, N = 32 queries), dK, dV of that half; S^T, dP^T over all of d
//
// Issue order per step i (one thread): dP_i, dV_i, S_{i+1}, dK_i, dQ_i, so the softmax-side
// work on step i+1's scores overlaps the tensor core's dK_i and dQ_i.
// Causal: a key tile only meets query tiles that reach its diagonal (whole tiles in the
// future are skipped, §5.3) and only pairs crossing the diagonal are masked element-wise.
#include <cuda.h>
#include <cuda_runtime.h>
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <vector>

#include "kernels.h"
#include "ptx.cuh"
#include "tmap.h"

namespace fa {
namespace {

constexpr int BN = 128;  // key rows per CTA

template <int D>
struct BwdCfg {
  // d = 256: a work item is one half of d of a key tile's outputs (dK, dV and dQ columns
  // [128 h, 128 h + 128)); both halves recompute S^T and dP^T over all 256 dimensions, since the
  // dV and dK accumulators of a whole row (2 x 256 columns) would fill all of TMEM
  static constexpr bool SPLITD = (D == 256);
  static constexpr int DH = SPLITD ? 128 : D;  // output columns of d per item
  static constexpr bool DQT = (D >= 128);      // dQ^T = K^T dS^T (TMEM lanes = d)
  static constexpr int BM = D == 64 ? 128 : (D == 128 ? 64 : 32);  // query rows per step
  static constexpr bool K_IN_TMEM = true;      // K_j as the TMEM A operand of S^T (d/2 columns)
  static constexpr bool DS_SW64 = (BM == 32);  // dS^T rows of 64 bytes: the 64-byte swizzle
  static constexpr int KB = D / 64;
  static constexpr int KV_BYTES = BN * D * 2;
  static constexpr int QT_BYTES = BM * D * 2;
  static constexpr int DS_BYTES = BN * BM * 2;
  static constexpr int STG_BYTES = BM * DH * 4;
  // WG0 and WG1 compute (half the queries of a step each; d = 256: WG0 alone, 32 queries), then
  // the drain warpgroup, the TMA producer warp and the MMA warp.
  static constexpr int COMPUTE_WGS = BM / 32 >= 2 ? 2 : 1;
  static constexpr int DRAIN_WARP0 = 4 * COMPUTE_WGS;  // first warp of the drain warpgroup
  static constexpr int PRODUCER_WARP = DRAIN_WARP0 + 4;
  static constexpr int MMA_WARP = PRODUCER_WARP + 1;
  static constexpr int THREADS = 32 * (MMA_WARP + 1);
  static constexpr uint32_t ITEM_READERS = 1 + 4 * COMPUTE_WGS + 4;  // MMA, compute and drain warps
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + KV_BYTES;
  static constexpr int QSTAGES = SPLITD ? 2 : 3;             // query-tile ring depth
  static constexpr int OFF_Q = OFF_V + KV_BYTES;                 // [QSTAGES]
  static constexpr int OFF_DO = OFF_Q + QSTAGES * QT_BYTES;      // [QSTAGES]
  static constexpr int OFF_DS = OFF_DO + QSTAGES * QT_BYTES;
  static constexpr int OFF_STG = OFF_DS + DS_BYTES;              // dQ staging tile
  static constexpr int OFF_VEC = OFF_STG + STG_BYTES;            // [QSTAGES] x (L2[BM], D[BM]) fp32
  static constexpr int OFF_BAR = OFF_VEC + QSTAGES * 2 * BM * 4;
  static constexpr int NBAR = 22;
  // after the barriers: TMEM base, abort flag, the two work-item slots
  static constexpr int SMEM = OFF_BAR + NBAR * 8 + 32;
  // masked variant: the CTA's step list after the barriers (an int count, then uint16 entries
  // (query head of the group << 12 | 128-row query block), rounded up to 8 entries)
  static constexpr int OFF_LIST = SMEM;
  static constexpr int list_bytes(int entries) { return 16 + 2 * ((entries + 7) & ~7); }
  static constexpr int SUB = 128 / BM;  // steps per 128-row query block
  static constexpr int COMPUTE_THREADS = 128 * COMPUTE_WGS;
  static constexpr int DRAIN_THREADS = 128;
  // TMEM columns between packed 32-query chunks of P^T / dS^T: each chunk keeps its packed
  // values inside its own 32 fp32 columns, so neither compute warpgroup writes over scores the
  // other has yet to read
  static constexpr int CH_COLS = 32;
  static constexpr int EPI_THREADS = 128;  // threads that read dK, dV out of TMEM (the drain warpgroup)
  // the staging tile also carries an item's dV and dK as 16-bit [128 rows][64 columns] boxes with
  // the 128-byte swizzle (d = 128: dV, then dK, two boxes each; d = 64: dV and dK side by side;
  // d = 256: one box at a time)
  static_assert(STG_BYTES >= (SPLITD ? 1 : 2) * BN * 128 && OFF_STG % 1024 == 0 && OFF_DS % 1024 == 0,
                "staging tile");
  static_assert(SMEM <= 232448, "shared memory");
  // TMEM columns: K_j as a 16-bit A operand (d/2 columns), S^T (P^T packed into
  // the first 16 of each 32-query chunk's columns), dP^T (dS^T likewise), the dQ partial and the
  // dV, dK accumulators (DH columns each)
  static constexpr uint32_t COL_K = SPLITD ? 384 : (DQT ? 0 : 448);
  static constexpr uint32_t COL_S = SPLITD ? 0 : (DQT ? 64 : 0);
  static constexpr uint32_t COL_DP = COL_S + BM;
  static constexpr uint32_t COL_DQ = COL_DP + BM;
  static constexpr uint32_t COL_DV = SPLITD ? 128 : (DQT ? 256 : 320);
  static constexpr uint32_t COL_DK = SPLITD ? 256 : 384;
  static_assert(COL_DK + DH <= 512 && COL_DQ + (DQT ? BM : D) <= COL_DV &&
                    (COL_K >= COL_DK + DH || COL_K + D / 2 <= COL_S), "TMEM columns");
};

enum BwdBar {
  B_KV = 0,
  B_QD_FULL = 1,   // [3]
  B_QD_EMPTY = 4,  // [3]
  B_S_FULL = 7,
  B_DP_FULL = 8,
  B_P_READY = 9,
  B_DS_READY = 10,
  B_DQ_FULL = 11,
  B_DQ_FREE = 12,
  B_ACC_FULL = 13,
  B_DRAIN = 14,
  B_KT_READY = 15,  // K_j copied into TMEM
  B_KV_EMPTY = 16,  // the tensor core no longer reads this item's K_j, V_j (persistent)
  B_ACC_EMPTY = 17, // this item's dK, dV have left TMEM (persistent)
  B_ITEM_FULL = 18,   // [2] the producer published the next work item in its slot
  B_ITEM_EMPTY = 20,  // [2] every consumer warp has read it
};

// TMEM column of the packed 16-bit A operand (P^T or dS^T) for MMA k-step kk (16 queries):
// chunk c of 32 queries starts at c * ch_cols, the start of the chunk's own 32 fp32 columns
__host__ __device__ constexpr uint32_t packed_col(int kk, int ch_cols) {
  return (uint32_t)((kk >> 1) * ch_cols + (kk & 1) * 8);
}

// advance a (query tile, query head) step cursor
__device__ __forceinline__ void step_next(int& ii, int& g, int tiles_per_head) {
  if (++ii == tiles_per_head) {
    ii = 0;
    ++g;
  }
}

// Work item of the persistent backward: one 128-key tile of one key/value head.
struct BwdItem {
  int kvh;          // key/value head
  int dh;           // d = 256: which half of d this item's outputs cover (0 or 1), else 0
  int k0;           // first key row
  int i_start;      // first query tile reaching this key tile's diagonal (causal), else 0
  int nsteps_head;  // query tiles per query head
  int nsteps;       // steps: (query head of the group, query tile) pairs
};

// Persistent: a CTA (one per SM) takes work items from a queue (a ticket counter in the
// workspace, items numbered heaviest first) until it is empty, so CTAs that finish early take
// more, whatever the cause.  It keeps its TMEM, barriers and rings between items: the next
// item's K_j, V_j load as soon as the tensor core no longer reads the current ones (kv_empty),
// and the current item's dK, dV leave TMEM through the staging tile (TMA stores) while the next
// item's first scores are computed; its first dV, dK GEMMs wait until they have (acc_empty).
// Every barrier phase runs on counters that continue across items.  The producer warp draws
// the tickets and publishes each item in a two-slot ring (item_full / item_empty).  The last
// CTA to finish sets the counter back to zero, ready for the next launch.
// Masked variant (block mask and/or window): one CTA per item; one warp lists, before the
// roles start, the (query head of the group, 128-row query block) pairs that can see the key
// tile (block-mask byte set and some pair inside the causal and window bounds); every role
// walks that list.
template <int D, bool BF16, bool MASKED>
__global__ void __launch_bounds__(BwdCfg<D>::THREADS, 1)
    bwd_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                  const __grid_constant__ CUtensorMap tm_dq, const __grid_constant__ CUtensorMap tm_dk,
                  const __grid_constant__ CUtensorMap tm_dv, const float* __restrict__ lse2,
                  const float* __restrict__ delta, int n, int npad, int bh_count, int ktiles, float scale,
                  int causal, int group, unsigned long long* err, int window,
                  const uint8_t* __restrict__ block_mask, int mask_heads, int heads, unsigned* __restrict__ sched,
                  int hgroup) {
  using C = BwdCfg<D>;
  constexpr int BM = C::BM;
  extern __shared__ __align__(1024) uint8_t smem[];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + C::NBAR);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* item_slot = reinterpret_cast<volatile int*>(tmem_slot + 2);  // [2]
  const ErrCtx ctx{err, abort_flag};

  const int qtiles = (n + BM - 1) / BM;
  // d = 256: two items per key tile (the two halves of d, adjacent in the order, so both read
  // the tile's K, V and the query-side streams while they are in L2)
  constexpr int kHalves = C::SPLITD ? 2 : 1;
  const int64_t total_items = (int64_t)bh_count * ktiles * kHalves;
  // work item -> key/value head and key tile: head-major (CTAs running together share Q/dO in
  // L2); causal: heaviest (first) key tiles first within groups of heads
  auto tile_of = [&](int item, int* kvh, int* kt) {
    if (causal) {
      grouped_work_item(item, bh_count, ktiles, hgroup, kvh, kt);
    } else {
      *kvh = item / ktiles;
      *kt = item - *kvh * ktiles;
    }
  };
  int* list_hdr = reinterpret_cast<int*>(smem + C::OFF_LIST);
  uint16_t* slist = reinterpret_cast<uint16_t*>(smem + C::OFF_LIST + 16);
  if constexpr (MASKED) {
    if (warp == C::PRODUCER_WARP) {
      int kvh, kt;
      tile_of((int)blockIdx.x / kHalves, &kvh, &kt);
      const int k0 = kt * BN;
      const int nblk = (n + 127) / 128;
      const int kmax = min(n, k0 + BN) - 1;
      int count = 0;
      for (int g = 0; g < group; ++g) {
        const int qh = kvh * group + g;
        const uint8_t* mcol = block_mask ? block_mask + (int64_t)(mask_heads > 1 ? qh % heads : 0) * nblk * nblk + kt
                                         : nullptr;
        for (int base = 0; base < nblk; base += 32) {
          const int qb = base + lane;
          bool v = qb < nblk;
          if (v) {
            const int qmin = qb * 128, qmax = min(n, qmin + 128) - 1;
            if (mcol) v = mcol[(int64_t)qb * nblk] != 0;
            if (causal) v = v && k0 <= qmax;
            if (window > 0) {
              v = v && qmin - kmax < window;
              if (!causal) v = v && k0 - qmax < window;
            }
          }
          const unsigned any = __ballot_sync(0xffffffffu, v);
          if (v) slist[count + __popc(any & ((1u << lane) - 1u))] = (uint16_t)((g << 12) | qb);
          count += __popc(any);
        }
      }
      if (lane == 0) list_hdr[0] = count;
    }
  }
  const float scale_log2 = scale * 1.4426950408889634f;

  if (threadIdx.x == 0) {
    if ((smem_u32(smem) & 1023u) != 0) report_error(err, DERR_BAD_SMEM_ALIGN, 1);
    *abort_flag = (smem_u32(smem) & 1023u) != 0;
    mbar_init(bar + B_KV, 1);
    for (int s = 0; s < C::QSTAGES; ++s) {
      mbar_init(bar + B_QD_FULL + s, 1);
      mbar_init(bar + B_QD_EMPTY + s, 1);
    }
    mbar_init(bar + B_S_FULL, 1);
    mbar_init(bar + B_DP_FULL, 1);
    mbar_init(bar + B_P_READY, C::COMPUTE_THREADS);
    mbar_init(bar + B_DS_READY, C::COMPUTE_THREADS);
    mbar_init(bar + B_DQ_FULL, 1);
    mbar_init(bar + B_DQ_FREE, C::DRAIN_THREADS);
    mbar_init(bar + B_ACC_FULL, 1);
    mbar_init(bar + B_DRAIN, 1);
    mbar_init(bar + B_KT_READY, 128);
    mbar_init(bar + B_KV_EMPTY, 1);
    mbar_init(bar + B_ACC_EMPTY, C::EPI_THREADS);
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar + B_ITEM_FULL + t, 1);
      mbar_init(bar + B_ITEM_EMPTY + t, C::ITEM_READERS);
    }
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

  auto item_at = [&](int item) {
    BwdItem w;
    int kt;
    tile_of(item / kHalves, &w.kvh, &kt);
    w.dh = C::SPLITD ? (item & 1) : 0;
    w.k0 = kt * BN;
    w.i_start = causal ? kt * (BN / BM) : 0;
    w.nsteps_head = qtiles - w.i_start;
    w.nsteps = MASKED ? list_hdr[0] * C::SUB : group * w.nsteps_head;
    return w;
  };
  // this CTA's r-th item, -1 when there is none.  Masked: the CTA's own item only.  Otherwise
  // one warp's read of the producer's slot r % 2; every consumer warp reads every slot once.
  // `good` turns false (and the item -1) when the bounded wait for the slot ran out.
  auto next_item = [&](int r, bool& good) {
    if constexpr (MASKED) {
      return r == 0 ? (int)blockIdx.x : -1;
    } else {
      const int t = r & 1;
      good = __all_sync(0xffffffffu, mbar_wait(bar + B_ITEM_FULL + t, (uint32_t)(r >> 1) & 1, ctx, 150)) && good;
      const int item = good ? item_slot[t] : -1;
      __syncwarp();
      if (lane == 0) mbar_arrive(bar + B_ITEM_EMPTY + t);
      return item;
    }
  };
  // step i of an item -> (query head within the group, first query row)
  auto step_rows = [&](const BwdItem& w, int i, int ii, int g, int* gm, int* q0) {
    if constexpr (MASKED) {
      const uint32_t e = slist[i / C::SUB];
      *gm = (int)(e >> 12);
      *q0 = (int)(e & 0xFFFu) * 128 + (i % C::SUB) * BM;
    } else {
      *gm = g;
      *q0 = (w.i_start + ii) * BM;
    }
  };
  // K_j rows -> TMEM (A operand of S^T = K Q^T): 16-byte chunks of the swizzled smem tile; row
  // rit of the tile, TMEM lane quarter lane_base
  auto k_to_tmem = [&](int rit, uint32_t lane_base) {
    const uint32_t sw = (uint32_t)(rit & 7);
#pragma unroll
    for (int kb = 0; kb < C::KB; ++kb) {
      const uint8_t* krow = smem + C::OFF_K + kb * (BN * 128) + rit * 128;
      uint32_t w[32];
#pragma unroll
      for (int ch = 0; ch < 8; ++ch) {
        const uint4 x = *reinterpret_cast<const uint4*>(krow + (((uint32_t)ch ^ sw) << 4));
        w[4 * ch] = x.x;
        w[4 * ch + 1] = x.y;
        w[4 * ch + 2] = x.z;
        w[4 * ch + 3] = x.w;
      }
      tmem_st32(tmem_addr(tbase, lane_base, C::COL_K + kb * 32), w);
    }
    tmem_wait_st();
  };
  // 32 columns of a dK / dV accumulator row -> 16-bit pairs (x f)
  auto load_acc32 = [&](uint32_t lane_base, uint32_t col, float f, uint32_t (&pk)[16]) {
    uint32_t r[32];
    tmem_ld32(tmem_addr(tbase, lane_base, col), r);
    tmem_wait_ld();
    reg_fence(r);
#pragma unroll
    for (int t = 0; t < 16; ++t) pk[t] = pack2<BF16>(__uint_as_float(r[2 * t]) * f, __uint_as_float(r[2 * t + 1]) * f);
  };
  // 32 columns (chunk c) of row `row` of a [128 rows][64 columns] 16-bit box with the 128-byte
  // swizzle, the layout of the dK / dV tensor maps' boxes
  auto stage_row32 = [&](uint8_t* box, int row, int c, const uint32_t (&pk)[16]) {
    uint8_t* rp = box + row * 128;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const uint32_t ch = (uint32_t)((c & 1) * 4 + u);
      *reinterpret_cast<uint4*>(rp + ((ch ^ (uint32_t)(row & 7)) << 4)) =
          make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
    }
  };

  if (warp == C::PRODUCER_WARP) {
    // ------------------------------------------------------------------ TMA producer
    if (start_ok && lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      tma_prefetch_desc(&tm_do);
      uint32_t qpos = 0;  // query-tile ring loads issued (all items)
      int kv_loads = 0;
      bool ok = true;
      for (int r = 0;; ++r) {
        int item;
        if constexpr (MASKED) {
          item = r == 0 ? (int)blockIdx.x : -1;
        } else {
          // draw a ticket and publish the item (or -1: the queue is empty) once both readers of
          // the slot's previous item have it
          if (r >= 2 && !(ok = mbar_wait(bar + B_ITEM_EMPTY + (r & 1), (uint32_t)((r - 2) >> 1) & 1, ctx, 114))) break;
          const unsigned ticket = atomicAdd(sched, 1u);
          item = ticket < (unsigned)total_items ? (int)ticket : -1;
          item_slot[r & 1] = item;
          mbar_arrive(bar + B_ITEM_FULL + (r & 1));
        }
        if (item < 0) break;
        const BwdItem w = item_at(item);
        if (!(ok = debug_check(w.kvh >= 0 && w.kvh < bh_count && w.k0 >= 0 && w.k0 < n, ctx, 160))) break;
        // K_j, V_j once the tensor core no longer reads the previous item's
        if (r > 0 && !(ok = mbar_wait(bar + B_KV_EMPTY, (r - 1) & 1, ctx, 113))) break;
        mbar_arrive_expect_tx(bar + B_KV, 2 * C::KV_BYTES);
        for (int kb = 0; kb < C::KB; ++kb) {
          tma_load_3d(smem + C::OFF_K + kb * (BN * 128), &tm_k, bar + B_KV, kb * 64, w.k0, w.kvh);
          tma_load_3d(smem + C::OFF_V + kb * (BN * 128), &tm_v, bar + B_KV, kb * 64, w.k0, w.kvh);
        }
        ++kv_loads;
        for (int i = 0, ii = 0, g = 0; i < w.nsteps; ++i, step_next(ii, g, w.nsteps_head)) {
          const int s = qpos % C::QSTAGES, use = qpos / C::QSTAGES;
          if (use > 0 && !(ok = mbar_wait(bar + B_QD_EMPTY + s, (use - 1) & 1, ctx, 110))) break;
          int gm, q0;
          step_rows(w, i, ii, g, &gm, &q0);
          const int qh = w.kvh * group + gm;
          // the L and D rows of the step lie inside the head's padded vectors
          if (!(ok = debug_check(gm >= 0 && gm < group && q0 >= 0 && q0 + BM <= npad, ctx, 161))) break;
          uint64_t* fb = bar + B_QD_FULL + s;
          mbar_arrive_expect_tx(fb, 2 * C::QT_BYTES + 2 * BM * 4);
          for (int kb = 0; kb < C::KB; ++kb) {
            tma_load_3d(smem + C::OFF_Q + s * C::QT_BYTES + kb * (BM * 128), &tm_q, fb, kb * 64, q0, qh);
            tma_load_3d(smem + C::OFF_DO + s * C::QT_BYTES + kb * (BM * 128), &tm_do, fb, kb * 64, q0, qh);
          }
          float* vec = reinterpret_cast<float*>(smem + C::OFF_VEC) + s * 2 * BM;
          bulk_load(vec, lse2 + (int64_t)qh * npad + q0, BM * 4, fb);
          bulk_load(vec + BM, delta + (int64_t)qh * npad + q0, BM * 4, fb);
          ++qpos;
        }
        if (!ok) break;
      }
      // drain: every copy this thread started must land before the CTA may exit
      ErrCtx nctx = ctx;
      int no_abort = 0;
      nctx.abort = &no_abort;
      if (kv_loads > 0) mbar_wait(bar + B_KV, (kv_loads - 1) & 1, nctx, 111);
      for (int64_t p = (int64_t)qpos - 1; p >= 0 && p >= (int64_t)qpos - C::QSTAGES; --p)
        mbar_wait(bar + B_QD_FULL + p % C::QSTAGES, (uint32_t)(p / C::QSTAGES) & 1, nctx, 112);
    }
    __syncwarp();
  } else if (warp == C::MMA_WARP) {
    // ------------------------------------------------------------------ MMA issuer
    // The whole warp runs this loop converged, so the smem descriptors are warp-uniform;
    // one elected lane issues every MMA and commit (a commit tracks its own lane's MMAs).
    if (start_ok) {
      const bool leader = elect_one_sync();
      const uint32_t idesc_s = make_idesc_f16(BN, BM, BF16, false, false);  // S^T, dP^T: M = keys, N = queries
      const uint32_t idesc_kv = make_idesc_f16(BN, C::DH, BF16, false, true);   // dV, dK: M = keys, N = d (half)
      const uint32_t idesc_q = C::DQT ? make_idesc_f16(C::DH, BM, BF16, true, true)  // dQ^T: M = d (half), N = queries
                                      : make_idesc_f16(BM, D, BF16, true, true);   // dQ: M = queries, N = d
      const uint32_t ks = smem_u32(smem + C::OFF_K), vs = smem_u32(smem + C::OFF_V);
      const uint32_t dss = smem_u32(smem + C::OFF_DS);
      auto qs_of = [&](int s) { return smem_u32(smem + C::OFF_Q + s * C::QT_BYTES); };
      auto dos_of = [&](int s) { return smem_u32(smem + C::OFF_DO + s * C::QT_BYTES); };
      auto wait = [&](uint64_t* b, uint32_t parity, uint32_t site) {
        return __all_sync(0xffffffffu, mbar_wait(b, parity, ctx, site));
      };
      auto commit = [&](uint64_t* b) {
        if (leader) umma_commit(b);
        __syncwarp();
      };
      // K-major operand rows of 128 bytes in 64-column blocks: offset of K-slice kk (16 wide)
      auto kmaj = [](int kk, int rows) { return (uint32_t)((kk * 16 / 64) * (rows * 128) + (kk * 16 % 64) * 2); };
      // S^T = K Q_i^T with K_j from TMEM (A) and Q_i K-major in smem (B); d = 256: K_j K-major
      // in smem as well
      auto issue_s = [&](uint32_t b) {
        uint64_t bd[D / 16];
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) bd[kk] = make_sdesc_sw128(b + kmaj(kk, BM), 16, 1024);
        if constexpr (C::K_IN_TMEM) {
          if (leader) {
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk)
              umma_ts(tbase + C::COL_S, tbase + C::COL_K + kk * 8, bd[kk], idesc_s, kk > 0);
          }
        } else {
          uint64_t ad[D / 16];
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) ad[kk] = make_sdesc_sw128(ks + kmaj(kk, BN), 16, 1024);
          if (leader) {
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) umma_ss(tbase + C::COL_S, ad[kk], bd[kk], idesc_s, kk > 0);
          }
        }
        __syncwarp();
      };
      bool ok = true;
      uint32_t gs = 0;  // steps issued (all items): ring slot and barrier phases
      for (int r = 0, item = next_item(0, ok); ok && item >= 0; item = next_item(++r, ok)) {
        const BwdItem w = item_at(item);
        // this item's K_j, V_j in shared memory and K_j in TMEM
        ok = wait(bar + B_KV, r & 1, 120);
        if (ok) ok = wait(bar + B_KT_READY, r & 1, 126);
        if (ok && w.nsteps > 0) {
          ok = wait(bar + B_QD_FULL + gs % C::QSTAGES, (gs / C::QSTAGES) & 1, 121);
          if (ok) {
            tc_fence_after();
            issue_s(qs_of(gs % C::QSTAGES));
            commit(bar + B_S_FULL);
          }
        }
        // the previous item's dK, dV must have left TMEM before this item's first dV, dK
        bool acc_free = (r == 0);
        for (int i = 0; ok && i < w.nsteps; ++i, ++gs) {
          const int s = gs % C::QSTAGES;
          const uint32_t g1 = gs + 1;
          const int s1 = g1 % C::QSTAGES;
          const uint32_t qs = qs_of(s), dos = dos_of(s);
          // dP^T_i = V dO_i^T (A: 128 keys x d, B: BM queries x d, both K-major in smem), issued
          // before the wait for P^T_i so that the tensor core works while the softmax side
          // finishes it.  Its columns (holding dS^T_{i-1}) were last read by dK_{i-1}: same
          // issuing thread, in order.
          {
            uint64_t ad[D / 16], bd[D / 16];
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              ad[kk] = make_sdesc_sw128(vs + kmaj(kk, BN), 16, 1024);
              bd[kk] = make_sdesc_sw128(dos + kmaj(kk, BM), 16, 1024);
            }
            if (leader) {
#pragma unroll
              for (int kk = 0; kk < D / 16; ++kk) umma_ss(tbase + C::COL_DP, ad[kk], bd[kk], idesc_s, kk > 0);
            }
            __syncwarp();
          }
          commit(bar + B_DP_FULL);
          // dV += P^T dO_i (P^T from TMEM, K = queries; dO_i as MN-major B: the item's DH columns,
          // 64-column boxes of BM rows)
          {
            uint64_t bd[BM / 16];
#pragma unroll
            for (int kk = 0; kk < BM / 16; ++kk)
              bd[kk] = make_sdesc_sw128(dos + w.dh * (C::DH / 64) * (BM * 128) + kk * 2048, BM * 128, 1024);
            if (!(ok = wait(bar + B_P_READY, gs & 1, 123))) break;
            if (!acc_free) {
              if (!(ok = wait(bar + B_ACC_EMPTY, (r - 1) & 1, 127))) break;
              acc_free = true;
            }
            tc_fence_after();
            if (leader) {
#pragma unroll
              for (int kk = 0; kk < BM / 16; ++kk)
                umma_ts(tbase + C::COL_DV, tbase + C::COL_S + packed_col(kk, C::CH_COLS), bd[kk], idesc_kv,
                        (i > 0 || kk > 0) ? 1u : 0u);
            }
            __syncwarp();
          }
          // S^T_{i+1}: overwrites P^T_i only after dV_i has read it (same issuing thread, in order)
          if (i + 1 < w.nsteps) {
            if (!(ok = wait(bar + B_QD_FULL + s1, (g1 / C::QSTAGES) & 1, 121))) break;
            tc_fence_after();
            issue_s(qs_of(s1));
            commit(bar + B_S_FULL);
          }
          // dK += dS^T Q_i (dS^T 16-bit in TMEM over the dP^T columns, Q_i MN-major B) and the dQ
          // partial (K and dS^T from smem; the previous partial, of this item or the last, drained
          // from TMEM first).  The dQ k-steps, whose A operand comes from shared memory, are
          // interleaved with the dK k-steps, whose A is in TMEM and which write another
          // accumulator: a shared-memory-A MMA then overlaps the other's arithmetic instead of
          // waiting for its operand reads, and the pair runs at about the tensor core's rate.
          // The first kDkHead dK k-steps go out before the wait for the drain.
          {
            uint64_t dk_b[BM / 16], kd[BN / 16], sd[BN / 16];
#pragma unroll
            for (int kk = 0; kk < BM / 16; ++kk)
              dk_b[kk] = make_sdesc_sw128(qs + w.dh * (C::DH / 64) * (BM * 128) + kk * 2048, BM * 128, 1024);
#pragma unroll
            for (int kk = 0; kk < BN / 16; ++kk) {
              // K as MN-major (d contiguous; the item's DH columns), dS^T as MN-major (queries
              // contiguous: 128-byte rows, or 64-byte rows with the 64-byte swizzle at d = 256)
              kd[kk] = make_sdesc_sw128(ks + w.dh * (C::DH / 64) * (BN * 128) + kk * 2048, BN * 128, 1024);
              if constexpr (C::DS_SW64)
                sd[kk] = make_sdesc_sw64(dss + kk * 1024, BN * 64, 512);
              else
                sd[kk] = make_sdesc_sw128(dss + kk * 2048, BN * 128, 1024);
            }
            constexpr int kDkHead = BM / 64;  // 1 at d = 128, 2 at d = 64, 0 at d = 256
            if (!(ok = wait(bar + B_DS_READY, gs & 1, 124))) break;
            tc_fence_after();
            if (leader) {
#pragma unroll
              for (int kk = 0; kk < kDkHead; ++kk)
                umma_ts(tbase + C::COL_DK, tbase + C::COL_DP + packed_col(kk, C::CH_COLS), dk_b[kk], idesc_kv,
                        (i > 0 || kk > 0) ? 1u : 0u);
            }
            __syncwarp();
            if (gs > 0) {
              if (!(ok = wait(bar + B_DQ_FREE, (gs - 1) & 1, 122))) break;
              tc_fence_after();
            }
            if (leader) {
              constexpr int NA = BN / 16, NB = BM / 16 - kDkHead;  // dQ and remaining dK k-steps
              int a = 0, b = 0;
#pragma unroll
              for (int t = 0; t < NA + NB; ++t) {
                if (b >= NB || (a < NA && a * NB <= b * NA)) {
                  const int kk = a++;
                  if constexpr (C::DQT)
                    umma_ss(tbase + C::COL_DQ, kd[kk], sd[kk], idesc_q, kk > 0);
                  else
                    umma_ss(tbase + C::COL_DQ, sd[kk], kd[kk], idesc_q, kk > 0);
                } else {
                  const int kk = kDkHead + b++;
                  umma_ts(tbase + C::COL_DK, tbase + C::COL_DP + packed_col(kk, C::CH_COLS), dk_b[kk], idesc_kv,
                          (i > 0 || kk > 0) ? 1u : 0u);
                  if (b == NB) umma_commit(bar + B_QD_EMPTY + s);  // Q_i, dO_i no longer read
                }
              }
              umma_commit(bar + B_DQ_FULL);
            }
            __syncwarp();
          }
        }
        // an item without steps still takes its turn on acc_empty, so the phases stay in step
        if (ok && !acc_free) ok = wait(bar + B_ACC_EMPTY, (r - 1) & 1, 127);
        if (ok) {
          commit(bar + B_ACC_FULL);  // this item's dK, dV accumulators are final
          commit(bar + B_KV_EMPTY);  // and its K_j, V_j are no longer read
        }
      }
      // drain: all MMAs complete before TMEM is released
      ErrCtx nctx = ctx;
      int no_abort = 0;
      nctx.abort = &no_abort;
      commit(bar + B_DRAIN);
      mbar_wait(bar + B_DRAIN, 0, nctx, 125);
    }
    __syncwarp();
  } else if (warp >= C::DRAIN_WARP0) {
    // ---------------------------------------------------------------- drain warpgroup: dQ, epilogue
    // Each dQ partial goes from TMEM to a staging tile in the layout of the dQ accumulator's
    // tensor map and one thread adds it to global memory (TMA reduce).  After an item's last
    // partial, its dV and dK (x tau) go through the same staging tile to global memory (TMA
    // stores), while the compute warpgroups start the next item.
    const uint32_t lane_base = (warp & 3) * 32;
    // TMEM lane: d index (d = 128; d = 256: within the item's half) or query row (d = 64) of a dQ
    // partial; key row of dK, dV
    const int rr = (warp & 3) * 32 + lane;
    const bool leader = (warp == C::DRAIN_WARP0 && lane == 0);
    uint8_t* stg = smem + C::OFF_STG;
    bool ok = start_ok;
    uint32_t gs = 0;  // dQ partials drained (all items)
    // Every warp runs every step of every item and passes every named barrier; once a bounded
    // wait has run out (the abort flag then ends every later wait at once) the warp still passes
    // them, staging stale TMEM columns that are never stored, so none is left waiting.  Whether
    // to take another item is decided by all four warps together (a reducing named barrier), so
    // they leave the loop at the same item.
    for (int r = 0;; ++r) {
      bool got = true;
      const int item = next_item(r, got);
      if (!named_bar_and(1, 128, got && item >= 0)) break;
      const BwdItem w = item_at(item);
      for (int i = 0, ii = 0, g = 0; i < w.nsteps; ++i, ++gs, step_next(ii, g, w.nsteps_head)) {
        int gm, q0;
        step_rows(w, i, ii, g, &gm, &q0);
        ok = __all_sync(0xffffffffu, mbar_wait(bar + B_DQ_FULL, gs & 1, ctx, 140)) && ok;
        tc_fence_after();
        constexpr int DQC = (C::DQT ? BM : D) / 32;  // 32-column TMEM chunks of a dQ partial
        uint32_t vr[DQC][32];
#pragma unroll
        for (int c = 0; c < DQC; ++c) tmem_ld32(tmem_addr(tbase, lane_base, C::COL_DQ + c * 32), vr[c]);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < DQC; ++c) reg_fence(vr[c]);
        const uint32_t* v = &vr[0][0];
        tc_fence_before();
        mbar_arrive(bar + B_DQ_FREE);
        if (leader) bulk_wait_group_read<0>();  // the previous bulk copy has finished reading the tile
        named_bar_sync(1, 128);
        if constexpr (C::DQT) {
          // [BM queries][DH] fp32, row-major: column rr (this thread's d) of each query row
          float* st = reinterpret_cast<float*>(stg) + rr;
#pragma unroll
          for (int q = 0; q < BM; ++q) st[q * C::DH] = __uint_as_float(v[q]);
        } else {
          // [BM queries][64] fp32 as two 128-byte-swizzled boxes of 32 columns: row rr (this
          // thread's query), 16-byte chunks
          const uint32_t sw = (uint32_t)(rr & 7);
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            uint8_t* bx = stg + (j >> 3) * (BM * 128) + rr * 128;
            *reinterpret_cast<uint4*>(bx + (((uint32_t)(j & 7) ^ sw) << 4)) =
                make_uint4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
          }
        }
        fence_proxy_async_smem();
        named_bar_sync(1, 128);
        if (leader && ok) {
          tma_reduce_add_3d(&tm_dq, stg, w.dh * C::DH, q0, w.kvh * group + gm);
          if constexpr (!C::DQT) tma_reduce_add_3d(&tm_dq, stg + BM * 128, 32, q0, w.kvh * group + gm);
          bulk_commit_group();
        }
      }
      // epilogue of this item: dV, dK rows rr -> 16-bit -> staging ([2 boxes][128 rows][64
      // columns], the layout of the dK / dV tensor maps) -> TMA stores (rows past N are not
      // written).  An item without steps (masked) stores zeros.
      ok = __all_sync(0xffffffffu, mbar_wait(bar + B_ACC_FULL, r & 1, ctx, 132)) && ok;
      const bool acc = ok && w.nsteps > 0;
      if (acc) tc_fence_after();
      if constexpr (C::SPLITD) {
        // d = 256: this row's DH columns of dV and of dK (x tau) into registers, the accumulators
        // released, then one 16 KB box at a time through the staging tile (dV's two, then dK's)
        uint32_t pvv[C::DH / 32][16], pkv[C::DH / 32][16];
#pragma unroll
        for (int c = 0; c < C::DH / 32; ++c) {
#pragma unroll
          for (int t = 0; t < 16; ++t) pvv[c][t] = pkv[c][t] = 0u;
          if (acc) {
            load_acc32(lane_base, C::COL_DV + c * 32, 1.f, pvv[c]);
            load_acc32(lane_base, C::COL_DK + c * 32, scale, pkv[c]);
          }
        }
        tc_fence_before();
        mbar_arrive(bar + B_ACC_EMPTY);  // the accumulators may be overwritten
#pragma unroll
        for (int t = 0; t < 2; ++t) {
#pragma unroll
          for (int b = 0; b < C::DH / 64; ++b) {
            if (leader) bulk_wait_group_read<0>();  // the previous bulk copy has read the tile
            named_bar_sync(1, 128);
            stage_row32(stg, rr, 0, t ? pkv[2 * b] : pvv[2 * b]);
            stage_row32(stg, rr, 1, t ? pkv[2 * b + 1] : pvv[2 * b + 1]);
            fence_proxy_async_smem();
            named_bar_sync(1, 128);
            if (leader && ok) {
              tma_store_3d(t ? &tm_dk : &tm_dv, stg, w.dh * C::DH + b * 64, w.k0, w.kvh);
              bulk_commit_group();
            }
          }
        }
      } else {
      uint32_t pkk[D / 2];  // this row of dK x tau, packed
      if (leader) bulk_wait_group_read<0>();  // the last dQ reduction has read the staging tile
      named_bar_sync(1, 128);
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t pv[16] = {};
        if (acc) load_acc32(lane_base, C::COL_DV + c * 32, 1.f, pv);
        stage_row32(stg + (c >> 1) * (BN * 128), rr, c, pv);
      }
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t pv[16] = {};
        if (acc) load_acc32(lane_base, C::COL_DK + c * 32, scale, pv);
#pragma unroll
        for (int t = 0; t < 16; ++t) pkk[c * 16 + t] = pv[t];
      }
      tc_fence_before();
      mbar_arrive(bar + B_ACC_EMPTY);  // the accumulators may be overwritten
      fence_proxy_async_smem();
      named_bar_sync(1, 128);
      if (leader) {
        if (ok) {
          for (int b = 0; b < D / 64; ++b) tma_store_3d(&tm_dv, stg + b * (BN * 128), b * 64, w.k0, w.kvh);
          bulk_commit_group();
        }
        bulk_wait_group_read<0>();
      }
      named_bar_sync(1, 128);
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t pv[16];
#pragma unroll
        for (int t = 0; t < 16; ++t) pv[t] = pkk[c * 16 + t];
        stage_row32(stg + (c >> 1) * (BN * 128), rr, c, pv);
      }
      fence_proxy_async_smem();
      named_bar_sync(1, 128);
      if (leader && ok) {
        for (int b = 0; b < D / 64; ++b) tma_store_3d(&tm_dk, stg + b * (BN * 128), b * 64, w.k0, w.kvh);
        bulk_commit_group();
      }
      }
    }
    if (leader) bulk_wait_group<0>();  // every reduction and store issued here has completed

  } else {
    {
      // ---------------------------------------------------------------- WG0, WG1: P^T, dS^T
      // Both warpgroups own the same 128 key rows (TMEM lane quarter warp % 4) and each takes
      // half of every step's 32-query chunks for P^T and dS^T.  WG0 also copies K_j into TMEM
      // at the start of an item.
      const int wg = warp >> 2;
      const uint32_t lane_base = (warp & 3) * 32;
      const int rit = (warp & 3) * 32 + lane;  // key row within the tile (and TMEM lane)
      uint8_t* ds_row = smem + C::OFF_DS + rit * 128;
      const uint32_t sw = (uint32_t)(rit & 7);
      constexpr int NCH = BM / (32 * C::COMPUTE_WGS);  // 32-query chunks a compute warpgroup takes
      const int c0 = wg * NCH;
      bool ok = start_ok;
      uint32_t gs = 0;  // steps processed (all items)
      for (int r = 0, item = next_item(0, ok); ok && item >= 0; item = next_item(++r, ok)) {
        const BwdItem w = item_at(item);
        const int key = w.k0 + rit;
        const bool key_ok = key < n;
        if (wg == 0) {
          // K_j -> TMEM: the previous item's last S^T (which read it) completed before its last step
          ok = __all_sync(0xffffffffu, mbar_wait(bar + B_KV, r & 1, ctx, 134));
          if (!ok) break;
          if constexpr (C::K_IN_TMEM) k_to_tmem(rit, lane_base);
          tc_fence_before();
          mbar_arrive(bar + B_KT_READY);
        }
        for (int i = 0, ii = 0, g = 0; ok && i < w.nsteps; ++i, ++gs, step_next(ii, g, w.nsteps_head)) {
          const int s = gs % C::QSTAGES;
          int gm, q0;
          step_rows(w, i, ii, g, &gm, &q0);
          const float* l2v = reinterpret_cast<const float*>(smem + C::OFF_VEC) + s * 2 * BM;
          const float* dvec = l2v + BM;
          // L_i, D_i arrive with the query tile (TMA); S^T_i from the tensor core
          ok = __all_sync(0xffffffffu, mbar_wait(bar + B_QD_FULL + s, (gs / C::QSTAGES) & 1, ctx, 133));
          if (ok) ok = __all_sync(0xffffffffu, mbar_wait(bar + B_S_FULL, gs & 1, ctx, 130));
          if (!ok) break;
          tc_fence_after();
          // visible queries q0 + qc: qc in [mask_below, mask_above) (causal: not before this key;
          // window: |query - key| < window, an upper bound on the query with or without causal)
          int mask_below = causal ? key - q0 : INT32_MIN, mask_above = INT32_MAX;
          if constexpr (MASKED) {
            if (window > 0) {
              mask_below = max(mask_below, key - window + 1 - q0);
              mask_above = key + window - q0;
            }
          }
          // the whole warp sees every query of the step: no masking of P
          const bool all_visible = __all_sync(0xffffffffu, key_ok && mask_below <= 0 && mask_above >= BM);
          // P^T of this key against this half's queries, kept as packed 16-bit pairs: the same
          // rounded values feed dV += P^T dO and dS = P o (dP - D)
          // One 32-query chunk at a time: its scores (TMEM) and, with two chunks (d = 64), its
          // -L log2 e values (shared memory) are loaded together, all in flight before one wait,
          // so no load's latency stands between two exponentials (GPT-2-medium backward 3 %
          // faster; with one chunk (d = 128) the preload measured 1.4 % slower).
          constexpr bool kPreload = NCH > 1;
          uint32_t pk[NCH * 16];
#pragma unroll
          for (int cl = 0; cl < NCH; ++cl) {
            const int c = c0 + cl;
            uint32_t r[32];
            tmem_ld32(tmem_addr(tbase, lane_base, C::COL_S + c * 32), r);
            float4 lc[kPreload ? 8 : 1];
            if constexpr (kPreload) {
#pragma unroll
              for (int u = 0; u < 8; ++u) lc[u] = *reinterpret_cast<const float4*>(l2v + c * 32 + 4 * u);
            }
            tmem_wait_ld();
            reg_fence(r);
            {
#pragma unroll
              for (int t = 0; t < 32; t += 4) {
                // x = S tau log2 e - L log2 e, two queries per paired FMA (l2v holds -L log2 e)
                const float4 l4 = kPreload ? lc[t / 4] : *reinterpret_cast<const float4*>(l2v + c * 32 + t);
                const float2 x01 = ffma2(make_float2(__uint_as_float(r[t]), __uint_as_float(r[t + 1])), scale_log2,
                                         make_float2(l4.x, l4.y));
                const float2 x23 = ffma2(make_float2(__uint_as_float(r[t + 2]), __uint_as_float(r[t + 3])),
                                         scale_log2, make_float2(l4.z, l4.w));
                float e[4] = {ex2(x01.x), ex2(x01.y), ex2(x23.x), ex2(x23.y)};
                if (!all_visible) {
#pragma unroll
                  for (int u = 0; u < 4; ++u) {
                    const int qc = c * 32 + t + u;
                    e[u] = (key_ok && qc >= mask_below && qc < mask_above) ? e[u] : 0.f;
                  }
                }
                pk[cl * 16 + t / 2] = pack2<BF16>(e[0], e[1]);
                pk[cl * 16 + t / 2 + 1] = pack2<BF16>(e[2], e[3]);
              }
            }
          }
#pragma unroll
          for (int cl = 0; cl < NCH; ++cl) {
            uint32_t wv[16];
#pragma unroll
            for (int t = 0; t < 16; ++t) wv[t] = pk[cl * 16 + t];
            tmem_st16(tmem_addr(tbase, lane_base, C::COL_S + (c0 + cl) * C::CH_COLS), wv);
          }
          tmem_wait_st();
          tc_fence_before();
          mbar_arrive(bar + B_P_READY);
          // dS^T = P^T o (dP^T - D); dp_full(i) also means the MMAs of step i-1 that read dS^T are done
          ok = __all_sync(0xffffffffu, mbar_wait(bar + B_DP_FULL, gs & 1, ctx, 131));
          if (!ok) break;
          tc_fence_after();
          {
            // one 32-query chunk at a time, its dP^T (TMEM) and (d = 64) D values loaded together;
            // a chunk's dS^T goes over the first 16 of its own 32 dP^T columns, so the next
            // chunk's dP^T is untouched
#pragma unroll
            for (int cl = 0; cl < NCH; ++cl) {
              const int c = c0 + cl;
              uint32_t r[32];
              tmem_ld32(tmem_addr(tbase, lane_base, C::COL_DP + c * 32), r);
              float4 dc[kPreload ? 8 : 1];
              if constexpr (kPreload) {
#pragma unroll
                for (int u = 0; u < 8; ++u) dc[u] = *reinterpret_cast<const float4*>(dvec + c * 32 + 4 * u);
              }
              tmem_wait_ld();
              reg_fence(r);
              uint32_t dsk[16];
#pragma unroll
              for (int t = 0; t < 16; t += 2) {
                // dS = P o (dP - D), two queries per paired subtract and multiply
                const float4 d4 = kPreload ? dc[t / 2] : *reinterpret_cast<const float4*>(dvec + c * 32 + 2 * t);
                const float2 ds01 = fmul2(unpack2<BF16>(pk[cl * 16 + t]),
                                          fsub2(make_float2(__uint_as_float(r[2 * t]), __uint_as_float(r[2 * t + 1])),
                                                make_float2(d4.x, d4.y)));
                const float2 ds23 =
                    fmul2(unpack2<BF16>(pk[cl * 16 + t + 1]),
                          fsub2(make_float2(__uint_as_float(r[2 * t + 2]), __uint_as_float(r[2 * t + 3])),
                                make_float2(d4.z, d4.w)));
                dsk[t] = pack2<BF16>(ds01.x, ds01.y);
                dsk[t + 1] = pack2<BF16>(ds23.x, ds23.y);
              }
              // 32 queries = 64 bytes = four 16-byte chunks of this key's row: 128-byte rows with
              // the 128-byte swizzle, or (32 queries a step) 64-byte rows with the 64-byte swizzle
              // (chunk index XOR bits 1-2 of the row)
              if constexpr (C::DS_SW64) {
                uint8_t* row64 = smem + C::OFF_DS + rit * 64;
                const uint32_t sw64 = (uint32_t)((rit >> 1) & 3);
#pragma unroll
                for (int u = 0; u < 4; ++u)
                  *reinterpret_cast<uint4*>(row64 + (((uint32_t)u ^ sw64) << 4)) =
                      make_uint4(dsk[4 * u], dsk[4 * u + 1], dsk[4 * u + 2], dsk[4 * u + 3]);
              } else {
                uint8_t* blk = ds_row + (c >> 1) * (BN * 128);
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                  const uint32_t ch = (uint32_t)((c & 1) * 4 + u);
                  *reinterpret_cast<uint4*>(blk + ((ch ^ sw) << 4)) =
                      make_uint4(dsk[4 * u], dsk[4 * u + 1], dsk[4 * u + 2], dsk[4 * u + 3]);
                }
              }
              // and packed into TMEM over this chunk's dP^T columns, already read (A operand of
              // dK += dS^T Q)
              tmem_st16(tmem_addr(tbase, lane_base, C::COL_DP + c * C::CH_COLS), dsk);
            }
          }
          fence_proxy_async_smem();
          tmem_wait_st();
          tc_fence_before();
          mbar_arrive(bar + B_DS_READY);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == C::MMA_WARP) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
  if constexpr (!MASKED) {
    // this CTA draws no more tickets; the last one to get here empties the queue for the next
    // launch (every CTA has drawn its last ticket by then)
    if (threadIdx.x == 0) {
      __threadfence();
      if (atomicAdd(sched + 1, 1u) == gridDim.x - 1) {
        atomicExch(sched, 0u);
        atomicExch(sched + 1, 0u);
      }
    }
  }
}

template <int D, bool BF16, bool MASKED>
cudaError_t launch_bwd_d(const BwdArgs& a) {
  using C = BwdCfg<D>;
  const int npad = (int)padded_rows(a.n);
  CUtensorMap tq, tk, tv, tdo, tdq, tdk, tdv;
  const int bh_kv = a.bh / a.group;
  if (!make_tmap_16bit_3d(&tq, a.q, BF16, D, a.n, a.bh, C::BM) || !make_tmap_16bit_3d(&tk, a.k, BF16, D, a.n, bh_kv, BN) ||
      !make_tmap_16bit_3d(&tv, a.v, BF16, D, a.n, bh_kv, BN) ||
      !make_tmap_16bit_3d(&tdo, a.dout, BF16, D, a.n, a.bh, C::BM) ||
      !make_tmap_f32_3d(&tdq, a.dq_acc, D, npad, a.bh, C::DQT ? C::DH : 32, C::BM, !C::DQT) ||
      !make_tmap_16bit_3d(&tdk, a.dk, BF16, D, a.n, bh_kv, BN) || !make_tmap_16bit_3d(&tdv, a.dv, BF16, D, a.n, bh_kv, BN))
    return cudaErrorInvalidValue;
  auto kern = bwd_tc_kernel<D, BF16, MASKED>;
  const int nblk = (a.n + 127) / 128;
  if (MASKED && !bwd_masked_fits(a.group, a.n, D)) return cudaErrorInvalidValue;
  const int smem = C::SMEM + (MASKED ? C::list_bytes(a.group * nblk) : 0);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int ktiles = (a.n + BN - 1) / BN;
  const int64_t items = (int64_t)bh_kv * ktiles * (C::SPLITD ? 2 : 1);
  const int64_t grid = MASKED ? items : std::min<int64_t>(items, device_sm_count());
  if (!MASKED && !a.sched) return cudaErrorInvalidValue;
  // causal order: groups of key/value heads whose query-side streams (Q, dO, the fp32 dQ
  // accumulator, L and D of each of their `group` query heads) stay in L2
  const int hgroup = head_group_for_l2((int64_t)a.group * ((int64_t)npad * D * 8 + (int64_t)npad * 8), kL2HeadBudgetBwd);
  kern<<<(unsigned)grid, C::THREADS, smem, a.stream>>>(tq, tk, tv, tdo, tdq, tdk, tdv, a.lse2, a.delta, a.n, npad,
                                                       bh_kv, ktiles, a.scale, a.causal, a.group, a.err, a.window,
                                                       a.block_mask, a.mask_heads, a.heads, a.sched, hgroup);
  return cudaGetLastError();
}

template <int D, bool BF16>
cudaError_t launch_bwd_dm(const BwdArgs& a) {
  return a.masked() ? launch_bwd_d<D, BF16, true>(a) : launch_bwd_d<D, BF16, false>(a);
}

}  // namespace

bool bwd_tc_supported(int dtype, int d) {
  return (dtype == DT_BF16 || dtype == DT_FP16) && (d == 64 || d == 128 || d == 256);
}

bool bwd_masked_fits(int group, int n, int d) {
  // step-list entries pack (query head of the group, 128-row block) into 16 bits, and the
  // list must fit in shared memory beside the kernel's tiles
  const int nblk = (n + 127) / 128;
  if (group > 16 || nblk > 4096) return false;
  const int smem = d == 256   ? BwdCfg<256>::SMEM + BwdCfg<256>::list_bytes(group * nblk)
                   : d == 128 ? BwdCfg<128>::SMEM + BwdCfg<128>::list_bytes(group * nblk)
                              : BwdCfg<64>::SMEM + BwdCfg<64>::list_bytes(group * nblk);
  return smem <= 232448;
}

cudaError_t launch_bwd_tc(const BwdArgs& a) {
  const bool bf = a.dtype == DT_BF16;
  switch (a.d) {
    case 64: return bf ? launch_bwd_dm<64, true>(a) : launch_bwd_dm<64, false>(a);
    case 128: return bf ? launch_bwd_dm<128, true>(a) : launch_bwd_dm<128, false>(a);
    case 256: return bf ? launch_bwd_dm<256, true>(a) : launch_bwd_dm<256, false>(a);
    default: return cudaErrorNotSupported;
  }
}

}  // namespace fa
