// Tensor-core backward for bf16/fp16, head dims 64/128 (sm_103a: TMA, tcgen05, TMEM).
//
// Recomputing backward ("Lecture 8 · GPU Performance & FlashAttention" §5.4; "FlashAttention
// and GPU memory" §09): nothing N x N was stored, so every (key tile j, query tile i) pair
// recomputes its scores from Q, K and the saved row statistic L:
//     S^T = K_j Q_i^T,   P^T = exp2(S^T tau log2e - L_i log2e)       (= e^(S - m)/l)
//     dV_j += P^T dO_i,   dP^T = V_j dO_i^T,   dS^T = P^T o (dP^T - D_i)
//     dK_j += dS^T Q_i,   dQ_i += dS K_j      (tau applied to dK here and to dQ on conversion)
// with D_i = sum_k dO_ik O_ik precomputed by the preprocess kernel (the §5.4 identity).
//
// One CTA owns a 128-key tile of one key/value head for its whole life (with grouped-query
// attention it visits every query head of that key/value head): K_j, V_j stay in shared
// memory and the dK_j, dV_j accumulators stay in TMEM, while query tiles (Q_i, dO_i, L_i,
// D_i) stream through a three-stage TMA ring.  Working transposed puts keys on TMEM lanes, so
// one thread owns one key row: P^T and dS^T need no cross-thread reduction.  K_j, P^T and
// dS^T sit in TMEM as A operands (S^T = K Q^T, dV += P^T dO, dK += dS^T Q), which spares
// the shared-memory read of A that an all-smem MMA pays; dS^T also goes to shared memory
// as an operand of the dQ GEMM.
//
// Two warpgroups share the elementwise work: both own the tile's 128 key rows (a warp reads
// the TMEM lanes of its quarter, so warps w and w + 4 see the same rows) and each takes half of
// every step's queries for P^T and dS^T.  dQ partials are summed over key tiles in an fp32
// accumulator in global memory: after its dS^T half, each warpgroup drains its half of the
// previous step's dQ partial from TMEM into a shared-memory staging tile, and one thread adds
// the tile to global memory with a TMA bulk reduction (whole 128-byte lines, no per-element
// atomics).  Two shapes of the dQ GEMM keep every TMEM region separate, so no
// GEMM waits for another region to be drained:
//   d = 64:  128 queries per step, dQ = dS K   (M = 128 queries, N = 64)
//   d = 128:  64 queries per step, dQ^T = K^T dS^T (M = 128 = d, N = 64 queries)
//
// Issue order per step i (one thread): dP_i, dV_i, S_{i+1}, dK_i, dQ_i, so the softmax-side
// work on step i+1's scores overlaps the tensor core's dK_i and dQ_i.
// Causal: a key tile only meets query tiles that reach its diagonal (whole tiles in the
// future are skipped, §5.3) and only pairs crossing the diagonal are masked element-wise.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cmath>
#include <cstdint>

#include "kernels.h"
#include "ptx.cuh"
#include "tmap.h"

namespace fa {
namespace {

constexpr int BN = 128;  // key rows per CTA

template <int D>
struct BwdCfg {
  static constexpr bool DQT = (D == 128);        // dQ^T = K^T dS^T (TMEM lanes = d)
  static constexpr int BM = DQT ? 64 : 128;      // query rows per step
  static constexpr int KB = D / 64;
  static constexpr int KV_BYTES = BN * D * 2;
  static constexpr int QT_BYTES = BM * D * 2;
  static constexpr int DS_BYTES = BN * BM * 2;
  static constexpr int STG_BYTES = BM * D * 4;
  static constexpr int THREADS = 320;            // WG0, WG1 (P/dS, dQ drain), TMA warp, MMA warp
  static constexpr int PRODUCER_WARP = 8;
  static constexpr int MMA_WARP = 9;
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + KV_BYTES;
  static constexpr int QSTAGES = 3;                          // query-tile ring depth
  static constexpr int OFF_Q = OFF_V + KV_BYTES;                 // [QSTAGES]
  static constexpr int OFF_DO = OFF_Q + QSTAGES * QT_BYTES;      // [QSTAGES]
  static constexpr int OFF_DS = OFF_DO + QSTAGES * QT_BYTES;
  static constexpr int OFF_STG = OFF_DS + DS_BYTES;              // dQ staging tile
  static constexpr int OFF_VEC = OFF_STG + STG_BYTES;            // [QSTAGES] x (L2[BM], D[BM]) fp32
  static constexpr int OFF_BAR = OFF_VEC + QSTAGES * 2 * BM * 4;
  static constexpr int NBAR = 18;
  static constexpr int SMEM = OFF_BAR + NBAR * 8 + 16;
  // masked variant: the CTA's step list after the barriers (an int count, then uint16 entries
  // (query head of the group << 12 | 128-row query block), rounded up to 8 entries)
  static constexpr int OFF_LIST = SMEM;
  static constexpr int list_bytes(int entries) { return 16 + 2 * ((entries + 7) & ~7); }
  static constexpr int SUB = 128 / BM;  // steps per 128-row query block
  // d = 64 (128 queries per step): both warpgroups compute P^T, dS^T (half the queries each)
  // and drain half of each dQ partial; d = 128 (tensor-bound): warpgroup 0 computes P^T, dS^T
  // and warpgroup 1 drains whole dQ partials as soon as they complete
  static constexpr bool SPLIT = !DQT;
  static constexpr int COMPUTE_THREADS = SPLIT ? 256 : 128;
  static constexpr int DRAIN_THREADS = SPLIT ? 256 : 128;
  static constexpr int CH_COLS = SPLIT ? 32 : 16;  // TMEM columns between packed 32-query chunks
  // TMEM columns: K_j as a 16-bit A operand (d/2 columns), S^T (P^T packed into the first 16
  // of each 32-query chunk's columns), dP^T (dS^T likewise), the dQ partial and the dV, dK
  // accumulators
  static constexpr uint32_t COL_K = DQT ? 0 : 448;
  static constexpr uint32_t COL_S = DQT ? 64 : 0;
  static constexpr uint32_t COL_DP = COL_S + BM;
  static constexpr uint32_t COL_DQ = COL_DP + BM;
  static constexpr uint32_t COL_DV = DQT ? 256 : 320;
  static constexpr uint32_t COL_DK = 384;
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
  B_STG_FREE = 16,  // dQ staging tile free (the previous reduction has read it)
  B_STG_FULL = 17,  // both warpgroups wrote their half of the staging tile
};

// TMEM column of the packed 16-bit A operand (P^T or dS^T) for MMA k-step kk (16 queries),
// chunk c of 32 queries starting at c * ch_cols: contiguous (16) when one warpgroup reads every
// score before writing any, or at the start of the chunk's own 32 fp32 columns (32) when two
// warpgroups share the queries, so neither writes over scores the other has yet to read
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

template <int D>
__device__ __forceinline__ void store_row16(void* base, int64_t row, const uint32_t (&pk)[16], int chunk) {
  uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(base) + row * D * 2 + chunk * 64);
#pragma unroll
  for (int i = 0; i < 4; ++i) dst[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
}

// Masked variant (block mask and/or window): one warp lists, before the roles start, the
// (query head of the group, 128-row query block) pairs that can see this key tile (block-mask
// byte set and some pair inside the causal and window bounds); every role walks that list.
template <int D, bool BF16, bool MASKED>
__global__ void __launch_bounds__(BwdCfg<D>::THREADS, 1)
    bwd_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                  const __grid_constant__ CUtensorMap tm_dq, const float* __restrict__ lse2,
                  const float* __restrict__ delta, void* __restrict__ dk_out, void* __restrict__ dv_out, int n,
                  int npad, int bh_count, int ktiles, float scale, int causal, int group, unsigned long long* err,
                  int window, const uint8_t* __restrict__ block_mask, int mask_heads, int heads) {
  using C = BwdCfg<D>;
  constexpr int BM = C::BM;
  extern __shared__ __align__(1024) uint8_t smem[];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + C::NBAR);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const ErrCtx ctx{err, abort_flag};

  // work item: head-major (CTAs running together share Q/dO in L2); causal: heaviest (first)
  // key tiles first within groups of heads
  int kvh, kt;  // key/value head and key tile of this CTA
  if (causal) {
    grouped_work_item(blockIdx.x, bh_count, ktiles, &kvh, &kt);
  } else {
    kvh = blockIdx.x / ktiles;
    kt = blockIdx.x - kvh * ktiles;
  }
  const int k0 = kt * BN;
  const int qtiles = (n + BM - 1) / BM;
  const int i_start = causal ? kt * (BN / BM) : 0;  // first query tile reaching this key tile's diagonal
  // steps: (query head of this key/value head's group, query tile) pairs; dK, dV sum over all
  const int nsteps_head = qtiles - i_start;
  int nsteps = group * nsteps_head;
  int* list_hdr = reinterpret_cast<int*>(smem + C::OFF_LIST);
  uint16_t* slist = reinterpret_cast<uint16_t*>(smem + C::OFF_LIST + 16);
  if constexpr (MASKED) {
    if (warp == C::PRODUCER_WARP) {
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
  // step i -> (query head within the group, first query row)
  auto step_rows = [&](int i, int ii, int g, int* gm, int* q0) {
    if constexpr (MASKED) {
      const uint32_t e = slist[i / C::SUB];
      *gm = (int)(e >> 12);
      *q0 = (int)(e & 0xFFFu) * 128 + (i % C::SUB) * BM;
    } else {
      *gm = g;
      *q0 = (i_start + ii) * BM;
    }
  };
  // each role walks the steps with a (query tile ii, query head g of the group) cursor, advanced
  // by step_next (no integer division on the per-step path)
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
    mbar_init(bar + B_STG_FREE, 1);
    mbar_init(bar + B_STG_FULL, C::DRAIN_THREADS);
    mbar_init(bar + B_ACC_FULL, 1);
    mbar_init(bar + B_DRAIN, 1);
    mbar_init(bar + B_KT_READY, 128);
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
  if constexpr (MASKED) nsteps = list_hdr[0] * C::SUB;

  if (warp == C::PRODUCER_WARP) {
    // ------------------------------------------------------------------ TMA producer
    if (start_ok && lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      tma_prefetch_desc(&tm_do);
      mbar_arrive_expect_tx(bar + B_KV, 2 * C::KV_BYTES);
      for (int kb = 0; kb < C::KB; ++kb) {
        tma_load_3d(smem + C::OFF_K + kb * (BN * 128), &tm_k, bar + B_KV, kb * 64, k0, kvh);
        tma_load_3d(smem + C::OFF_V + kb * (BN * 128), &tm_v, bar + B_KV, kb * 64, k0, kvh);
      }
      int issued = 0;
      for (int i = 0, ii = 0, g = 0; i < nsteps; ++i, step_next(ii, g, nsteps_head)) {
        const int s = i % C::QSTAGES, use = i / C::QSTAGES;
        if (use > 0 && !mbar_wait(bar + B_QD_EMPTY + s, (use - 1) & 1, ctx, 110)) break;
        int gm, q0;
        step_rows(i, ii, g, &gm, &q0);
        const int qh = kvh * group + gm;
        uint64_t* fb = bar + B_QD_FULL + s;
        mbar_arrive_expect_tx(fb, 2 * C::QT_BYTES + 2 * BM * 4);
        for (int kb = 0; kb < C::KB; ++kb) {
          tma_load_3d(smem + C::OFF_Q + s * C::QT_BYTES + kb * (BM * 128), &tm_q, fb, kb * 64, q0, qh);
          tma_load_3d(smem + C::OFF_DO + s * C::QT_BYTES + kb * (BM * 128), &tm_do, fb, kb * 64, q0, qh);
        }
        float* vec = reinterpret_cast<float*>(smem + C::OFF_VEC) + s * 2 * BM;
        bulk_load(vec, lse2 + (int64_t)qh * npad + q0, BM * 4, fb);
        bulk_load(vec + BM, delta + (int64_t)qh * npad + q0, BM * 4, fb);
        issued = i + 1;
      }
      ErrCtx nctx = ctx;
      int no_abort = 0;
      nctx.abort = &no_abort;
      mbar_wait(bar + B_KV, 0, nctx, 111);
      for (int i = issued - 1; i >= 0 && i >= issued - C::QSTAGES; --i)
        mbar_wait(bar + B_QD_FULL + i % C::QSTAGES, (i / C::QSTAGES) & 1, nctx, 112);
    }
    __syncwarp();
  } else if (warp == C::MMA_WARP) {
    // ------------------------------------------------------------------ MMA issuer
    // The whole warp runs this loop converged, so the smem descriptors are warp-uniform;
    // one elected lane issues every MMA and commit (a commit tracks its own lane's MMAs).
    if (start_ok) {
      const bool leader = elect_one_sync();
      const uint32_t idesc_s = make_idesc_f16(BN, BM, BF16, false, false);  // S^T, dP^T: M = keys, N = queries
      const uint32_t idesc_kv = make_idesc_f16(BN, D, BF16, false, true);   // dV, dK: M = keys, N = d
      const uint32_t idesc_q = C::DQT ? make_idesc_f16(D, BM, BF16, true, true)    // dQ^T: M = d, N = queries
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
      // dP^T = V dO_i^T (A: 128 keys x d, B: BM queries x d, both K-major in smem)
      auto issue_dp = [&](uint32_t b) {
        uint64_t ad[D / 16], bd[D / 16];
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          ad[kk] = make_sdesc_sw128(vs + kmaj(kk, BN), 16, 1024);
          bd[kk] = make_sdesc_sw128(b + kmaj(kk, BM), 16, 1024);
        }
        if (leader) {
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) umma_ss(tbase + C::COL_DP, ad[kk], bd[kk], idesc_s, kk > 0);
        }
        __syncwarp();
      };
      // S^T = K Q_i^T with K_j from TMEM (A) and Q_i K-major in smem (B)
      auto issue_s = [&](uint32_t b) {
        uint64_t bd[D / 16];
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) bd[kk] = make_sdesc_sw128(b + kmaj(kk, BM), 16, 1024);
        if (leader) {
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) umma_ts(tbase + C::COL_S, tbase + C::COL_K + kk * 8, bd[kk], idesc_s, kk > 0);
        }
        __syncwarp();
      };
      bool ok = wait(bar + B_KV, 0, 120);
      if (ok) ok = wait(bar + B_KT_READY, 0, 126);
      if (ok && nsteps > 0) {
        ok = wait(bar + B_QD_FULL + 0, 0, 121);
        if (ok) {
          tc_fence_after();
          issue_s(qs_of(0));
          commit(bar + B_S_FULL);
        }
      }
      for (int i = 0; ok && i < nsteps; ++i) {
        const int s = i % C::QSTAGES;
        const int s1 = (i + 1) % C::QSTAGES;
        const uint32_t qs = qs_of(s), dos = dos_of(s);
        // dP^T_i (its columns, holding dS^T_{i-1}, were last read by dK_{i-1}: same lane, in order)
        issue_dp(dos);
        commit(bar + B_DP_FULL);
        // dV += P^T dO_i (P^T from TMEM, K = queries; dO_i as MN-major B)
        {
          uint64_t bd[BM / 16];
#pragma unroll
          for (int kk = 0; kk < BM / 16; ++kk) bd[kk] = make_sdesc_sw128(dos + kk * 2048, BM * 128, 1024);
          if (!(ok = wait(bar + B_P_READY, i & 1, 123))) break;
          tc_fence_after();
          if (leader) {
#pragma unroll
            for (int kk = 0; kk < BM / 16; ++kk)
              umma_ts(tbase + C::COL_DV, tbase + C::COL_S + packed_col(kk, C::CH_COLS), bd[kk], idesc_kv, (i > 0 || kk > 0) ? 1u : 0u);
          }
          __syncwarp();
        }
        // S^T_{i+1}: overwrites P^T_i only after dV_i has read it (same issuing lane, in order)
        if (i + 1 < nsteps) {
          if (!(ok = wait(bar + B_QD_FULL + s1, ((i + 1) / C::QSTAGES) & 1, 121))) break;
          tc_fence_after();
          issue_s(qs_of(s1));
          commit(bar + B_S_FULL);
        }
        // dK += dS^T Q_i (dS^T 16-bit in TMEM over the dP^T columns, Q_i MN-major)
        {
          uint64_t bd[BM / 16];
#pragma unroll
          for (int kk = 0; kk < BM / 16; ++kk) bd[kk] = make_sdesc_sw128(qs + kk * 2048, BM * 128, 1024);
          if (!(ok = wait(bar + B_DS_READY, i & 1, 124))) break;
          tc_fence_after();
          if (leader) {
#pragma unroll
            for (int kk = 0; kk < BM / 16; ++kk)
              umma_ts(tbase + C::COL_DK, tbase + C::COL_DP + packed_col(kk, C::CH_COLS), bd[kk], idesc_kv, (i > 0 || kk > 0) ? 1u : 0u);
          }
          __syncwarp();
        }
        commit(bar + B_QD_EMPTY + s);
        // dQ partial (the previous one drained from TMEM first)
        {
          uint64_t kd[BN / 16], sd[BN / 16];
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk) {
            kd[kk] = make_sdesc_sw128(ks + kk * 2048, BN * 128, 1024);   // K as MN-major (d contiguous)
            sd[kk] = make_sdesc_sw128(dss + kk * 2048, BN * 128, 1024);  // dS^T as MN-major (queries contiguous)
          }
          if (i > 0) {
            if (!(ok = wait(bar + B_DQ_FREE, (i - 1) & 1, 122))) break;
            tc_fence_after();
          }
          if (leader) {
#pragma unroll
            for (int kk = 0; kk < BN / 16; ++kk) {
              if constexpr (C::DQT)
                umma_ss(tbase + C::COL_DQ, kd[kk], sd[kk], idesc_q, kk > 0);
              else
                umma_ss(tbase + C::COL_DQ, sd[kk], kd[kk], idesc_q, kk > 0);
            }
          }
          __syncwarp();
        }
        commit(bar + B_DQ_FULL);
      }
      if (ok) commit(bar + B_ACC_FULL);
      // drain: all MMAs complete before TMEM is released
      ErrCtx nctx = ctx;
      int no_abort = 0;
      nctx.abort = &no_abort;
      commit(bar + B_DRAIN);
      mbar_wait(bar + B_DRAIN, 0, nctx, 125);
    }
    __syncwarp();
  } else if (!C::SPLIT && warp < 4) {
    // ---------------------------------------------------------------- WG0: P^T, dS^T, epilogue
    const uint32_t lane_base = warp * 32;
    const int rit = warp * 32 + lane;  // key row within the tile
    const int key = k0 + rit;
    const bool key_ok = key < n;
    uint8_t* ds_row = smem + C::OFF_DS + rit * 128;
    const uint32_t sw = (uint32_t)(rit & 7);
    bool ok = start_ok;
    // K_j row -> TMEM (A operand of S^T = K Q^T): 16-byte chunks of the swizzled smem tile
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(bar + B_KV, 0, ctx, 134));
    if (ok) {
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
      tc_fence_before();
      mbar_arrive(bar + B_KT_READY);
    }
    for (int i = 0, ii = 0, g = 0; ok && i < nsteps; ++i, step_next(ii, g, nsteps_head)) {
      const int s = i % C::QSTAGES;
      int gm, q0;
      step_rows(i, ii, g, &gm, &q0);
      const float* l2v = reinterpret_cast<const float*>(smem + C::OFF_VEC) + s * 2 * BM;
      const float* dvec = l2v + BM;
      // L_i, D_i arrive with the query tile (TMA); S^T_i from the tensor core
      ok = __all_sync(0xffffffffu, mbar_wait(bar + B_QD_FULL + s, (i / C::QSTAGES) & 1, ctx, 133));
      if (ok) ok = __all_sync(0xffffffffu, mbar_wait(bar + B_S_FULL, i & 1, ctx, 130));
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
      // P^T row (this key against the BM queries), kept as packed 16-bit pairs: the same
      // rounded values feed dV += P^T dO and dS = P o (dP - D)
      uint32_t pk[BM / 2];
#pragma unroll
      for (int g = 0; g < BM / 64; ++g) {  // 64 columns per batch of TMEM loads
      uint32_t sr[2][32];
      tmem_ld32(tmem_addr(tbase, lane_base, C::COL_S + g * 64), sr[0]);
      tmem_ld32(tmem_addr(tbase, lane_base, C::COL_S + g * 64 + 32), sr[1]);
      tmem_wait_ld();
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        const int c = g * 2 + cc;
        uint32_t(&r)[32] = sr[cc];
        reg_fence(r);
#pragma unroll
        for (int t = 0; t < 32; t += 4) {
          const float4 l4 = *reinterpret_cast<const float4*>(l2v + c * 32 + t);
          const float lv[4] = {l4.x, l4.y, l4.z, l4.w};
          float e[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int qc = c * 32 + t + u;
            const float x = ex2(fmaf(__uint_as_float(r[t + u]), scale_log2, -lv[u]));
            e[u] = (key_ok && qc >= mask_below && qc < mask_above) ? x : 0.f;
          }
          pk[(c * 32 + t) / 2] = pack2<BF16>(e[0], e[1]);
          pk[(c * 32 + t) / 2 + 1] = pack2<BF16>(e[2], e[3]);
        }
      }
      }
#pragma unroll
      for (int h = 0; h < BM / 64; ++h) {
        uint32_t w[32];
#pragma unroll
        for (int t = 0; t < 32; ++t) w[t] = pk[h * 32 + t];
        tmem_st32(tmem_addr(tbase, lane_base, C::COL_S + h * 32), w);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar + B_P_READY);
      // dS^T = P^T o (dP^T - D); dp_full(i) also means the MMAs of step i-1 that read dS^T are done
      ok = __all_sync(0xffffffffu, mbar_wait(bar + B_DP_FULL, i & 1, ctx, 131));
      if (!ok) break;
      tc_fence_after();
#pragma unroll
      for (int g = 0; g < BM / 64; ++g) {  // 64 columns per batch of TMEM loads
      uint32_t dr[2][32];
      tmem_ld32(tmem_addr(tbase, lane_base, C::COL_DP + g * 64), dr[0]);
      tmem_ld32(tmem_addr(tbase, lane_base, C::COL_DP + g * 64 + 32), dr[1]);
      tmem_wait_ld();
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        const int c = g * 2 + cc;
        uint32_t(&r)[32] = dr[cc];
        reg_fence(r);
        uint32_t dsk[16];
#pragma unroll
        for (int t = 0; t < 16; t += 2) {
          const float4 d4 = *reinterpret_cast<const float4*>(dvec + c * 32 + 2 * t);
          const float2 p01 = unpack2<BF16>(pk[c * 16 + t]);
          const float2 p23 = unpack2<BF16>(pk[c * 16 + t + 1]);
          dsk[t] = pack2<BF16>(p01.x * (__uint_as_float(r[2 * t]) - d4.x), p01.y * (__uint_as_float(r[2 * t + 1]) - d4.y));
          dsk[t + 1] = pack2<BF16>(p23.x * (__uint_as_float(r[2 * t + 2]) - d4.z),
                                   p23.y * (__uint_as_float(r[2 * t + 3]) - d4.w));
        }
        // 32 queries = 64 bytes = four 16-byte chunks of this key's row, 128-byte swizzle
        uint8_t* blk = ds_row + (c >> 1) * (BN * 128);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const uint32_t ch = (uint32_t)((c & 1) * 4 + u);
          *reinterpret_cast<uint4*>(blk + ((ch ^ sw) << 4)) =
              make_uint4(dsk[4 * u], dsk[4 * u + 1], dsk[4 * u + 2], dsk[4 * u + 3]);
        }
        // and packed into TMEM over dP^T columns already read (A operand of dK += dS^T Q)
        tmem_st16(tmem_addr(tbase, lane_base, C::COL_DP + c * 16), dsk);
      }
      }
      fence_proxy_async_smem();
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar + B_DS_READY);
    }
    // epilogue: dV, dK (x tau) from TMEM to global
    if (ok && nsteps > 0) {
      ok = __all_sync(0xffffffffu, mbar_wait(bar + B_ACC_FULL, 0, ctx, 132));
      if (ok) {
        tc_fence_after();
#pragma unroll 1
        for (int which = 0; which < 2; ++which) {
          const uint32_t col = which ? C::COL_DK : C::COL_DV;
          const float f = which ? scale : 1.f;
          void* dst = which ? dk_out : dv_out;
#pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            uint32_t r[32];
            tmem_ld32(tmem_addr(tbase, lane_base, col + c * 32), r);
            tmem_wait_ld();
            reg_fence(r);
            uint32_t pk[16];
#pragma unroll
            for (int t = 0; t < 16; ++t)
              pk[t] = pack2<BF16>(__uint_as_float(r[2 * t]) * f, __uint_as_float(r[2 * t + 1]) * f);
            if (key_ok) store_row16<D>(dst, (int64_t)kvh * n + key, pk, c);
          }
        }
      }
    } else if (ok && nsteps == 0 && key_ok) {
      // no query meets this key tile: zero gradients (not reachable for square causal masks)
      uint32_t pk[16] = {};
      for (int c = 0; c < D / 32; ++c) {
        store_row16<D>(dk_out, (int64_t)kvh * n + key, pk, c);
        store_row16<D>(dv_out, (int64_t)kvh * n + key, pk, c);
      }
    }

  } else if (!C::SPLIT && warp < 8) {
    // TMEM lane = d index (DQT) or query row; the partial goes to a staging tile in the layout
    // of the dQ accumulator's tensor map and one thread adds it to global memory (TMA reduce).
    const uint32_t lane_base = (warp & 3) * 32;
    const int rr = (warp & 3) * 32 + lane;
    const bool leader = (warp == 4 && lane == 0);
    bool ok = start_ok;
    // Every warp runs every step and passes both named barriers in each; once a bounded wait
    // has run out (the abort flag then ends every later wait at once) the warp still passes
    // them, staging stale TMEM columns that are never reduced, so none is left waiting.
    for (int i = 0, ii = 0, g = 0; i < nsteps; ++i, step_next(ii, g, nsteps_head)) {
      int gm, q0;
      step_rows(i, ii, g, &gm, &q0);
      ok = __all_sync(0xffffffffu, mbar_wait(bar + B_DQ_FULL, i & 1, ctx, 140)) && ok;
      tc_fence_after();
      uint32_t vr[2][32];
#pragma unroll
      for (int c = 0; c < 2; ++c) tmem_ld32(tmem_addr(tbase, lane_base, C::COL_DQ + c * 32), vr[c]);
      tmem_wait_ld();
      reg_fence(vr[0]);
      reg_fence(vr[1]);
      const uint32_t* v = &vr[0][0];
      tc_fence_before();
      mbar_arrive(bar + B_DQ_FREE);
      uint8_t* stg = smem + C::OFF_STG;
      if (leader) bulk_wait_group_read<0>();  // the previous reduction has finished reading the tile
      named_bar_sync(1, 128);
      if constexpr (C::DQT) {
        // [BM queries][D] fp32, row-major: column rr (this thread's d) of each query row
        float* st = reinterpret_cast<float*>(stg) + rr;
#pragma unroll
        for (int q = 0; q < BM; ++q) st[q * D] = __uint_as_float(v[q]);
      } else {
        // [128 queries][64] fp32 as two 128-byte-swizzled boxes of 32 columns; row rr
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          uint8_t* bx = stg + (j >> 3) * (BM * 128) + rr * 128;
          *reinterpret_cast<uint4*>(bx + (((uint32_t)(j & 7) ^ (uint32_t)(rr & 7)) << 4)) =
              make_uint4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
        }
      }
      fence_proxy_async_smem();
      named_bar_sync(1, 128);
      if (leader && ok) {
        const int qh = kvh * group + gm;
        if constexpr (C::DQT) {
          tma_reduce_add_3d(&tm_dq, stg, 0, q0, qh);
        } else {
          tma_reduce_add_3d(&tm_dq, stg, 0, q0, qh);
          tma_reduce_add_3d(&tm_dq, stg + BM * 128, 32, q0, qh);
        }
        bulk_commit_group();
      }
    }
    if (leader) bulk_wait_group<0>();  // every reduction issued here has completed

  } else if (warp < 8) {
    if constexpr (C::SPLIT) {
      // ---------------------------------------------------------------- WG0, WG1: P^T, dS^T, dQ drain
      // (d = 64, 128 queries per step) Both warpgroups own the same 128 key rows (TMEM lane
      // quarter warp % 4) and each takes half of every step's 32-query chunks for P^T and dS^T;
      // after its dS^T half of step i each drains its half of the dQ partial of step i - 1 (that
      // MMA completed before dP^T_i, which the dS^T half has just read).  WG0 also copies K_j
      // into TMEM at the start and writes dK, dV at the end.
      constexpr bool SPLIT = C::SPLIT;
      const int wg = warp >> 2;
      const uint32_t lane_base = (warp & 3) * 32;
      const int rit = (warp & 3) * 32 + lane;  // key row within the tile (and TMEM lane)
      const int key = k0 + rit;
      const bool key_ok = key < n;
      uint8_t* ds_row = smem + C::OFF_DS + rit * 128;
      const uint32_t sw = (uint32_t)(rit & 7);
      constexpr int NCH = SPLIT ? BM / 64 : BM / 32;  // 32-query chunks a computing warpgroup takes
      const int c0 = SPLIT ? wg * NCH : 0;
      constexpr int DCOLS = SPLIT ? 32 : 64;  // TMEM columns of a dQ partial one thread drains
      const int dcol0 = SPLIT ? wg * 32 : 0;
      const bool leader = (warp == (SPLIT ? 0 : 4) && lane == 0);  // issues the dQ reductions
      uint8_t* stg = smem + C::OFF_STG;
      bool ok = start_ok;
      if (wg == 0) {
        // K_j row -> TMEM (A operand of S^T = K Q^T): 16-byte chunks of the swizzled smem tile
        if (ok) ok = __all_sync(0xffffffffu, mbar_wait(bar + B_KV, 0, ctx, 134));
        if (ok) {
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
          tc_fence_before();
          mbar_arrive(bar + B_KT_READY);
        }
      }
      // dQ partial k -> staging tile (this warpgroup's half) -> one TMA reduce-add into the fp32
      // accumulator.  The staging handshake uses mbarriers (bounded waits), not named barriers,
      // so a warp that gave up cannot leave the others waiting.
      auto drain = [&](int k, int q0, int qh) {
        bool good = __all_sync(0xffffffffu, mbar_wait(bar + B_DQ_FULL, k & 1, ctx, 140));
        if (!good) return false;
        tc_fence_after();
        uint32_t vr[DCOLS / 32][32];  // this thread's TMEM columns of the partial
#pragma unroll
        for (int c = 0; c < DCOLS / 32; ++c) tmem_ld32(tmem_addr(tbase, lane_base, C::COL_DQ + dcol0 + c * 32), vr[c]);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < DCOLS / 32; ++c) reg_fence(vr[c]);
        const uint32_t* v = &vr[0][0];
        tc_fence_before();
        mbar_arrive(bar + B_DQ_FREE);
        if (leader) {
          bulk_wait_group_read<0>();  // the previous reduction has finished reading the tile
          mbar_arrive(bar + B_STG_FREE);
        }
        good = __all_sync(0xffffffffu, mbar_wait(bar + B_STG_FREE, k & 1, ctx, 141));
        if (!good) return false;
        if constexpr (C::DQT) {
          // [BM queries][D] fp32 row-major; TMEM lane = d (rit), columns = this thread's queries
          float* st = reinterpret_cast<float*>(stg) + rit;
#pragma unroll
          for (int qq = 0; qq < DCOLS; ++qq) st[(dcol0 + qq) * D] = __uint_as_float(v[qq]);
        } else {
          // [128 queries][64] fp32 as two 128-byte-swizzled boxes of 32 columns; TMEM lane =
          // query row (rit), columns = this thread's d (one box per 32)
#pragma unroll
          for (int j = 0; j < DCOLS / 4; ++j) {
            uint8_t* bx = stg + (dcol0 / 32 + j / 8) * (BM * 128) + rit * 128;
            *reinterpret_cast<uint4*>(bx + (((uint32_t)(j & 7) ^ sw) << 4)) =
                make_uint4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
          }
        }
        fence_proxy_async_smem();
        mbar_arrive(bar + B_STG_FULL);
        if (leader) {
          if (!mbar_wait(bar + B_STG_FULL, k & 1, ctx, 142)) return false;
          if constexpr (C::DQT) {
            tma_reduce_add_3d(&tm_dq, stg, 0, q0, qh);
          } else {
            tma_reduce_add_3d(&tm_dq, stg, 0, q0, qh);
            tma_reduce_add_3d(&tm_dq, stg + BM * 128, 32, q0, qh);
          }
          bulk_commit_group();
        }
        return true;
      };
      int prev_q0 = 0, prev_qh = 0;
      for (int i = 0, ii = 0, g = 0; ok && i < nsteps; ++i, step_next(ii, g, nsteps_head)) {
        const int s = i % C::QSTAGES;
        int gm, q0;
        step_rows(i, ii, g, &gm, &q0);

        const float* l2v = reinterpret_cast<const float*>(smem + C::OFF_VEC) + s * 2 * BM;
        const float* dvec = l2v + BM;
        // L_i, D_i arrive with the query tile (TMA); S^T_i from the tensor core
        ok = __all_sync(0xffffffffu, mbar_wait(bar + B_QD_FULL + s, (i / C::QSTAGES) & 1, ctx, 133));
        if (ok) ok = __all_sync(0xffffffffu, mbar_wait(bar + B_S_FULL, i & 1, ctx, 130));
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
        // P^T of this key against this half's queries, kept as packed 16-bit pairs: the same
        // rounded values feed dV += P^T dO and dS = P o (dP - D)
        uint32_t pk[NCH * 16];
        {
          uint32_t sr[NCH][32];
#pragma unroll
          for (int cl = 0; cl < NCH; ++cl) tmem_ld32(tmem_addr(tbase, lane_base, C::COL_S + (c0 + cl) * 32), sr[cl]);
          tmem_wait_ld();
#pragma unroll
          for (int cl = 0; cl < NCH; ++cl) {
            const int c = c0 + cl;
            uint32_t(&r)[32] = sr[cl];
            reg_fence(r);
#pragma unroll
            for (int t = 0; t < 32; t += 4) {
              const float4 l4 = *reinterpret_cast<const float4*>(l2v + c * 32 + t);
              const float lv[4] = {l4.x, l4.y, l4.z, l4.w};
              float e[4];
#pragma unroll
              for (int u = 0; u < 4; ++u) {
                const int qc = c * 32 + t + u;
                const float x = ex2(fmaf(__uint_as_float(r[t + u]), scale_log2, -lv[u]));
                e[u] = (key_ok && qc >= mask_below && qc < mask_above) ? x : 0.f;
              }
              pk[cl * 16 + t / 2] = pack2<BF16>(e[0], e[1]);
              pk[cl * 16 + t / 2 + 1] = pack2<BF16>(e[2], e[3]);
            }
          }
        }
#pragma unroll
        for (int cl = 0; cl < NCH; ++cl) {
          uint32_t w[16];
#pragma unroll
          for (int t = 0; t < 16; ++t) w[t] = pk[cl * 16 + t];
          tmem_st16(tmem_addr(tbase, lane_base, C::COL_S + (c0 + cl) * C::CH_COLS), w);
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(bar + B_P_READY);
        // dS^T = P^T o (dP^T - D); dp_full(i) also means the MMAs of step i-1 that read dS^T are done
        ok = __all_sync(0xffffffffu, mbar_wait(bar + B_DP_FULL, i & 1, ctx, 131));
        if (!ok) break;
        tc_fence_after();
        {
          uint32_t dr[NCH][32];
#pragma unroll
          for (int cl = 0; cl < NCH; ++cl) tmem_ld32(tmem_addr(tbase, lane_base, C::COL_DP + (c0 + cl) * 32), dr[cl]);
          tmem_wait_ld();
#pragma unroll
          for (int cl = 0; cl < NCH; ++cl) {
            const int c = c0 + cl;
            uint32_t(&r)[32] = dr[cl];
            reg_fence(r);
            uint32_t dsk[16];
#pragma unroll
            for (int t = 0; t < 16; t += 2) {
              const float4 d4 = *reinterpret_cast<const float4*>(dvec + c * 32 + 2 * t);
              const float2 p01 = unpack2<BF16>(pk[cl * 16 + t]);
              const float2 p23 = unpack2<BF16>(pk[cl * 16 + t + 1]);
              dsk[t] = pack2<BF16>(p01.x * (__uint_as_float(r[2 * t]) - d4.x),
                                   p01.y * (__uint_as_float(r[2 * t + 1]) - d4.y));
              dsk[t + 1] = pack2<BF16>(p23.x * (__uint_as_float(r[2 * t + 2]) - d4.z),
                                       p23.y * (__uint_as_float(r[2 * t + 3]) - d4.w));
            }
            // 32 queries = 64 bytes = four 16-byte chunks of this key's row, 128-byte swizzle
            uint8_t* blk = ds_row + (c >> 1) * (BN * 128);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const uint32_t ch = (uint32_t)((c & 1) * 4 + u);
              *reinterpret_cast<uint4*>(blk + ((ch ^ sw) << 4)) =
                  make_uint4(dsk[4 * u], dsk[4 * u + 1], dsk[4 * u + 2], dsk[4 * u + 3]);
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
        if constexpr (SPLIT) {
          if (i > 0 && !(ok = drain(i - 1, prev_q0, prev_qh))) break;
        }
        prev_q0 = q0;
        prev_qh = kvh * group + gm;
      }
      if (SPLIT && ok && nsteps > 0) ok = drain(nsteps - 1, prev_q0, prev_qh);
      if (leader) bulk_wait_group<0>();  // every reduction issued here has completed
      // epilogue (WG0): dV, dK (x tau) from TMEM to global
      if (wg == 0 && ok && nsteps > 0) {
        ok = __all_sync(0xffffffffu, mbar_wait(bar + B_ACC_FULL, 0, ctx, 132));
        if (ok) {
          tc_fence_after();
#pragma unroll 1
          for (int which = 0; which < 2; ++which) {
            const uint32_t col = which ? C::COL_DK : C::COL_DV;
            const float f = which ? scale : 1.f;
            void* dst = which ? dk_out : dv_out;
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
              uint32_t r[32];
              tmem_ld32(tmem_addr(tbase, lane_base, col + c * 32), r);
              tmem_wait_ld();
              reg_fence(r);
              uint32_t pk[16];
#pragma unroll
              for (int t = 0; t < 16; ++t)
                pk[t] = pack2<BF16>(__uint_as_float(r[2 * t]) * f, __uint_as_float(r[2 * t + 1]) * f);
              if (key_ok) store_row16<D>(dst, (int64_t)kvh * n + key, pk, c);
            }
          }
        }
      } else if (wg == 0 && ok && nsteps == 0 && key_ok) {
        // no query meets this key tile: zero gradients (not reachable for square causal masks)
        uint32_t pk[16] = {};
        for (int c = 0; c < D / 32; ++c) {
          store_row16<D>(dk_out, (int64_t)kvh * n + key, pk, c);
          store_row16<D>(dv_out, (int64_t)kvh * n + key, pk, c);
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
}

template <int D, bool BF16, bool MASKED>
cudaError_t launch_bwd_d(const BwdArgs& a) {
  using C = BwdCfg<D>;
  const int npad = (int)padded_rows(a.n);
  CUtensorMap tq, tk, tv, tdo, tdq;
  const int bh_kv = a.bh / a.group;
  if (!make_tmap_16bit_3d(&tq, a.q, BF16, D, a.n, a.bh, C::BM) || !make_tmap_16bit_3d(&tk, a.k, BF16, D, a.n, bh_kv, BN) ||
      !make_tmap_16bit_3d(&tv, a.v, BF16, D, a.n, bh_kv, BN) ||
      !make_tmap_16bit_3d(&tdo, a.dout, BF16, D, a.n, a.bh, C::BM) ||
      !make_tmap_f32_3d(&tdq, a.dq_acc, D, npad, a.bh, C::DQT ? D : 32, C::BM, !C::DQT))
    return cudaErrorInvalidValue;
  auto kern = bwd_tc_kernel<D, BF16, MASKED>;
  const int nblk = (a.n + 127) / 128;
  if (MASKED && !bwd_masked_fits(a.group, a.n, D)) return cudaErrorInvalidValue;
  const int smem = C::SMEM + (MASKED ? C::list_bytes(a.group * nblk) : 0);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int ktiles = (a.n + BN - 1) / BN;
  kern<<<(unsigned)(bh_kv * ktiles), C::THREADS, smem, a.stream>>>(tq, tk, tv, tdo, tdq, a.lse2, a.delta, a.dk, a.dv,
                                                                   a.n, npad, bh_kv, ktiles, a.scale, a.causal, a.group,
                                                                   a.err, a.window, a.block_mask, a.mask_heads,
                                                                   a.heads);
  return cudaGetLastError();
}

template <int D, bool BF16>
cudaError_t launch_bwd_dm(const BwdArgs& a) {
  return a.masked() ? launch_bwd_d<D, BF16, true>(a) : launch_bwd_d<D, BF16, false>(a);
}

}  // namespace

bool bwd_tc_supported(int dtype, int d) { return (dtype == DT_BF16 || dtype == DT_FP16) && (d == 64 || d == 128); }

bool bwd_masked_fits(int group, int n, int d) {
  // step-list entries pack (query head of the group, 128-row block) into 16 bits, and the
  // list must fit in shared memory beside the kernel's tiles
  const int nblk = (n + 127) / 128;
  if (group > 16 || nblk > 4096) return false;
  const int smem = (d == 128 ? BwdCfg<128>::SMEM + BwdCfg<128>::list_bytes(group * nblk)
                             : BwdCfg<64>::SMEM + BwdCfg<64>::list_bytes(group * nblk));
  return smem <= 232448;
}

cudaError_t launch_bwd_tc(const BwdArgs& a) {
  const bool bf = a.dtype == DT_BF16;
  switch (a.d) {
    case 64: return bf ? launch_bwd_dm<64, true>(a) : launch_bwd_dm<64, false>(a);
    case 128: return bf ? launch_bwd_dm<128, true>(a) : launch_bwd_dm<128, false>(a);
    default: return cudaErrorNotSupported;
  }
}

}  // namespace fa
