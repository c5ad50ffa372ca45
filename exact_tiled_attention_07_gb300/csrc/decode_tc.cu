// Tensor-core split-KV decode for bf16/fp16, head dims 64/128/256 (sm_103a: TMA, tcgen05, TMEM).
//
// What it computes: for the new query rows of one key/value head (every query head of the
// group, every new position) attention over the whole cache, O = softmax(tau Q K^T) V and
// L = m + ln l, with the cache cut into pieces that run in parallel and are merged with the
// online-softmax merge ("Lecture 8 · GPU Performance & FlashAttention" §8.2 split-KV decoding,
// Exercise 3 merge; §8.2 grouped-query attention for the shared key/value head).
//
// The rows that share a key/value head are contiguous in Q [B][H][Nq][d] (heads kvh*group ..
// kvh*group + group - 1, all Nq positions), so they form one 128-row query tile, which the
// softmax warps copy into TMEM once (lanes past the group's rows hold zeros); S = Q K_j^T then
// takes Q from TMEM and K_j from shared memory.  A CTA owns one (batch, key/value head,
// 128-row tile, piece of the cache); a piece is a run of whole key tiles (128 keys, 64 at
// d = 256).  Every cached key and value is read from HBM once per row tile, so the kernel is
// HBM-bound: the whole of shared memory is a K/V ring (14/7/7 stages at d = 64/128/256) that
// keeps the bytes in flight, and S is double-buffered in TMEM so the softmax of tile j + 1
// runs while the tensor core does P_j V_j and S_{j+2}.
//
// Few rows (the usual decode step: group x Nq <= 32 or <= 64): the rows are copied R = 4 or 2
// times into the four 32-lane quarters of the tile, and copy c takes only key columns
// [c*BN/R, (c+1)*BN/R) of every tile, the others' P set to zero.  Each copy is then an
// independent piece of the keys with its own running maximum, sum and O accumulator (the
// same split the pieces of the cache use), so the exponentials of a tile are spread over
// four warps instead of one; the copies are merged in shared memory at the end.
//
// Roles (192 threads): warps 0-3 softmax (one thread per TMEM lane), warp 4 TMA producer,
// warp 5 MMA issuer.  The online softmax is the forward kernel's (exp2 domain, lazy rescale
// by 2^8).  Output: with one piece, O (16-bit) and L; otherwise the piece's normalised O
// (fp32) and base-2 log-sum-exp m + log2 l into the workspace, folded by decode_merge.
#include <cuda.h>
#include <cuda_runtime.h>
#include <algorithm>
#include <cmath>
#include <cstdint>

#include "kernels.h"
#include "ptx.cuh"
#include "tmap.h"

namespace fa {
namespace {

constexpr int BM = 128;      // query rows per tile (TMEM lanes)
constexpr float kRescaleThreshold = 8.0f;
constexpr int kMaxDynamicSmem = 232448;  // 227 KB per CTA
constexpr int kMergeBarrier = 1;         // named barrier of the four softmax warps

template <int D>
struct DecCfg {
  static constexpr int BN = (D == 256) ? 64 : 128;  // keys per tile
  static constexpr int KB = D / 64;                 // 64-column (128-byte) blocks per row
  static constexpr int TILE_BYTES = BN * D * 2;
  static constexpr int STAGES_FIT = (kMaxDynamicSmem - 1024) / TILE_BYTES;
  static constexpr int STAGES = STAGES_FIT > 14 ? 14 : STAGES_FIT;
  static constexpr int PRODUCER_WARP = 4;
  static constexpr int MMA_WARP = 5;
  static constexpr int THREADS = 192;
  // TMEM columns: S double buffer, O accumulator, Q (16-bit pairs, the A operand of S = Q K^T)
  static constexpr int S_COL0 = 0, S_COL1 = BN, O_COL = 256;
  static constexpr int Q_COL = (D == 256) ? 2 * BN : O_COL + D;
  static_assert(Q_COL + D / 2 <= 512 && (Q_COL >= O_COL + D || Q_COL + D / 2 <= O_COL), "TMEM columns");
  // shared memory: the K/V ring only
  static constexpr int OFF_RING = 0;
  static constexpr int OFF_BAR = OFF_RING + STAGES * TILE_BYTES;
  static constexpr int NBAR = 1 + 2 * STAGES + 2 + 2 + 1 + 1 + 1;
  static constexpr int SMEM = OFF_BAR + NBAR * 8 + 16;
  // merge of the row copies, in the ring once every MMA is done: m, l [128] and O [128][D + 4]
  static constexpr int OROW = D + 4;
  static constexpr int MERGE_BYTES = (2 * BM + BM * OROW) * 4;
  static_assert(STAGES >= 2, "ring needs two stages");
  static_assert(SMEM <= kMaxDynamicSmem, "shared memory");
  static_assert(MERGE_BYTES <= STAGES * TILE_BYTES, "merge buffer fits in the ring");
};

template <int D, bool BF16, int R>
__global__ void __launch_bounds__(DecCfg<D>::THREADS, 1)
    decode_tc_kernel(const uint32_t* __restrict__ q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, void* __restrict__ out, float* __restrict__ lse,
                     float* __restrict__ ws_o, float* __restrict__ ws_l, int rows, int rows_per_batch, int hkv,
                     int row_tiles, int splits, int nk, float scale_log2, unsigned long long* err,
                     unsigned long long* counter) {
  using C = DecCfg<D>;
  constexpr int BN = C::BN;
  constexpr int QUARTERS = 4 / R;  // lane quarters per copy
  constexpr int COLS = BN / R;     // key columns of a tile taken by one copy
  static_assert(COLS % 32 == 0, "a copy takes whole 32-column groups");
  extern __shared__ __align__(1024) uint8_t smem[];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* q_full = bars;  // Q rows stored into TMEM by the four softmax warps
  uint64_t* kv_full = bars + 1;
  uint64_t* kv_empty = bars + 1 + C::STAGES;
  uint64_t* s_full = bars + 1 + 2 * C::STAGES;  // [2]
  uint64_t* p_full = s_full + 2;                // [2]: one per S buffer, so the softmax can never
                                                // run two phases ahead of the MMA warp's wait
  uint64_t* o_full = p_full + 2;
  uint64_t* pv_done = o_full + 1;
  uint64_t* drain = pv_done + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::NBAR);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const ErrCtx ctx{err, abort_flag};

  // work item: piece fastest, then row tile, then (batch, key/value head)
  int t = blockIdx.x;
  const int split = t % splits;
  t /= splits;
  const int rt = t % row_tiles;
  const int bkv = t / row_tiles;  // b * hkv + kvh: the key/value head in K, V
  const int b = bkv / hkv, kvh = bkv - b * hkv;
  const int64_t row_base = (int64_t)b * rows_per_batch + (int64_t)kvh * rows;  // first Q row of the group
  const int r0 = rt * BM;                                                       // first row of this tile
  const int mc = min(BM, rows - r0);                                            // rows of this tile
  // softmax warps holding at least one row of the tile (all four when R > 1)
  const int active_warps = R * min(QUARTERS, (mc + 31) / 32);
  const int tiles = (nk + BN - 1) / BN;
  const int j0 = (int)((int64_t)tiles * split / splits);
  const int nb = (int)((int64_t)tiles * (split + 1) / splits) - j0;  // key tiles of this piece

  if (threadIdx.x == 0) {
    if ((smem_u32(smem) & 1023u) != 0) report_error(err, DERR_BAD_SMEM_ALIGN, 0);
    *abort_flag = (smem_u32(smem) & 1023u) != 0;
    mbar_init(q_full, 128);
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(kv_full + s, 1);
      mbar_init(kv_empty + s, 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(s_full + i, 1);
      mbar_init(p_full + i, 32 * active_warps);
    }
    mbar_init(o_full, 1);
    mbar_init(pv_done, 1);
    mbar_init(drain, 1);
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
    if (start_ok && nb > 0 && lane == 0) {
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      int issued = 0;
      for (int idx = 0; idx < 2 * nb; ++idx) {
        const int slot = idx % C::STAGES, use = idx / C::STAGES;
        if (use > 0 && !mbar_wait(kv_empty + slot, (use - 1) & 1, ctx, 110)) break;
        mbar_arrive_expect_tx(kv_full + slot, C::TILE_BYTES);
        uint8_t* dst = smem + C::OFF_RING + slot * C::TILE_BYTES;
        const CUtensorMap* tm = (idx & 1) ? &tm_v : &tm_k;
        for (int kb = 0; kb < C::KB; ++kb)
          tma_load_3d(dst + kb * (BN * 128), tm, kv_full + slot, kb * 64, (j0 + (idx >> 1)) * BN, bkv);
        issued = idx + 1;
      }
      // drain: every copy this thread started must land before the CTA may exit
      ErrCtx nctx = ctx;
      int no_abort = 0;
      nctx.abort = &no_abort;
      for (int idx = issued - 1; idx >= 0 && idx >= issued - C::STAGES; --idx)
        mbar_wait(kv_full + idx % C::STAGES, (idx / C::STAGES) & 1, nctx, 112);
    }
    __syncwarp();
  } else if (warp == C::MMA_WARP) {
    // ------------------------------------------------------------------ MMA issuer
    // converged warp, one elected lane issues every MMA and commit
    if (start_ok && nb > 0) {
      const bool leader = elect_one_sync();
      const uint32_t idesc_qk = make_idesc_f16(BM, BN, BF16, false, false);
      const uint32_t idesc_pv = make_idesc_f16(BM, D, BF16, false, true);
      const uint32_t ring = smem_u32(smem + C::OFF_RING);
      auto slot_of = [&](int idx) { return idx % C::STAGES; };
      auto wait = [&](uint64_t* bar, uint32_t parity, uint32_t site) {
        return __all_sync(0xffffffffu, mbar_wait(bar, parity, ctx, site));
      };
      auto wait_full = [&](int idx) { return wait(kv_full + slot_of(idx), (idx / C::STAGES) & 1, 120); };
      auto commit = [&](uint64_t* bar) {
        if (leader) umma_commit(bar);
        __syncwarp();
      };
      // S = Q K_j^T into TMEM columns s_col (Q from TMEM, K_j from the ring)
      auto issue_qk = [&](int kidx, uint32_t s_col) {
        const uint32_t kt = ring + slot_of(kidx) * C::TILE_BYTES;
        uint64_t bd[D / 16];
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const int k0 = kk * 16;
          bd[kk] = make_sdesc_sw128(kt + (k0 / 64) * (BN * 128) + (k0 % 64) * 2, 16, 1024);
        }
        if (leader) {
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            umma_ts(tbase + s_col, tbase + C::Q_COL + kk * 8, bd[kk], idesc_qk, kk > 0 ? 1u : 0u);
        }
        __syncwarp();
      };
      // O += P V_j with P (16-bit pairs) in TMEM columns [p_col, p_col + BN / 2)
      auto issue_pv = [&](uint32_t p_col, int vidx, bool acc) {
        const uint32_t vt = ring + slot_of(vidx) * C::TILE_BYTES;
        uint64_t bd[BN / 16];
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk) bd[kk] = make_sdesc_sw128(vt + kk * 2048, BN * 128, 1024);
        if (leader) {
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk)
            umma_ts(tbase + C::O_COL, tbase + p_col + kk * 8, bd[kk], idesc_pv, (acc || kk > 0) ? 1u : 0u);
        }
        __syncwarp();
      };
      bool ok = wait(q_full, 0, 121);
      if (ok) tc_fence_after();
      for (int j = 0; ok && j < 2 && j < nb; ++j) {
        if (!(ok = wait_full(2 * j))) break;
        tc_fence_after();
        issue_qk(2 * j, j ? C::S_COL1 : C::S_COL0);
        commit(s_full + j);
        commit(kv_empty + slot_of(2 * j));
      }
      for (int j = 0; ok && j < nb; ++j) {
        const int vidx = 2 * j + 1;
        const uint32_t buf = (j & 1) ? C::S_COL1 : C::S_COL0;
        if (!(ok = wait_full(vidx))) break;
        if (!(ok = wait(p_full + (j & 1), (j >> 1) & 1, 122))) break;
        tc_fence_after();
        issue_pv(buf, vidx, j > 0);
        commit(pv_done);
        commit(kv_empty + slot_of(vidx));
        if (j + 2 < nb) {
          const int kidx = 2 * (j + 2);
          if (!(ok = wait_full(kidx))) break;
          tc_fence_after();
          issue_qk(kidx, buf);  // in order after P_j V_j, which reads this buffer
          commit(s_full + (j & 1));
          commit(kv_empty + slot_of(kidx));
        }
        if (j == nb - 1) commit(o_full);
      }
      // drain: all MMAs complete before TMEM is released
      ErrCtx nctx = ctx;
      int no_abort = 0;
      nctx.abort = &no_abort;
      commit(drain);
      mbar_wait(drain, 0, nctx, 125);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------ softmax (one TMEM lane per thread)
    constexpr int QR = BM / R;                      // rows per copy
    const int cp = warp / QUARTERS;                 // copy: key columns [cp * COLS, (cp + 1) * COLS)
    const int rit = (warp % QUARTERS) * 32 + lane;  // row within the tile
    const uint32_t lane_base = warp * 32;
    const int col0 = cp * COLS;
    const bool warp_active = (warp % QUARTERS) * 32 < mc;
    const bool valid = rit < mc;
    float m = -INFINITY;  // reference maximum of this copy, log2 units
    float l = 0.f;
    bool ok = start_ok;
    if (ok && nb > 0) {
      // this lane's Q row into TMEM as 16-bit pairs (element 2c in the low half of column c);
      // lanes past the tile's rows get zeros
      const uint32_t* qrow = q + (row_base + r0 + rit) * (D / 2);
#pragma unroll 1
      for (int c = 0; c < D / 64; ++c) {
        uint32_t w[32];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const uint4 u = valid ? reinterpret_cast<const uint4*>(qrow + c * 32)[i] : make_uint4(0u, 0u, 0u, 0u);
          w[4 * i] = u.x;
          w[4 * i + 1] = u.y;
          w[4 * i + 2] = u.z;
          w[4 * i + 3] = u.w;
        }
        tmem_st32(tmem_addr(tbase, lane_base, C::Q_COL + c * 32), w);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(q_full);
    }
    for (int j = 0; warp_active && ok && j < nb; ++j) {
      const uint32_t s_col = (j & 1) ? C::S_COL1 : C::S_COL0;
      ok = __all_sync(0xffffffffu, mbar_wait(s_full + (j & 1), (j >> 1) & 1, ctx, 130));
      if (!ok) break;
      tc_fence_after();
      uint32_t sr[COLS / 32][32];
#pragma unroll
      for (int c = 0; c < COLS / 32; ++c) tmem_ld32(tmem_addr(tbase, lane_base, s_col + col0 + c * 32), sr[c]);
      tmem_wait_ld();
#pragma unroll
      for (int c = 0; c < COLS / 32; ++c) reg_fence(sr[c]);
      float s[COLS];
#pragma unroll
      for (int c = 0; c < COLS / 32; ++c)
#pragma unroll
        for (int i = 0; i < 32; ++i) s[c * 32 + i] = __uint_as_float(sr[c][i]);
      // keys past the end of the cache (last tile only)
      const int limit = nk - (j0 + j) * BN - col0;
      if (limit < COLS) {
#pragma unroll
        for (int c = 0; c < COLS; ++c)
          if (c >= limit) s[c] = -INFINITY;
      }
      const float mx = row_max(s);
      const float m_blk = mx * scale_log2;
      float alpha = 1.f;
      bool rescale = false;
      if (m == -INFINITY) {
        m = m_blk;  // first block with a visible key for this copy (O is still zero)
        alpha = 0.f;
      } else if (m_blk > m + kRescaleThreshold) {
        alpha = ex2(m - m_blk);
        m = m_blk;
        rescale = true;
      }
      const float neg_m = (m == -INFINITY) ? 0.f : -m;
      float part[4] = {0.f, 0.f, 0.f, 0.f};  // four partial sums: no single long add chain
      // this copy's P: 16-bit pairs, COLS / 2 TMEM columns from column col0 / 2 of the buffer
#pragma unroll
      for (int h = 0; h < COLS / 32; ++h) {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float p0 = ex2(fmaf(s[h * 32 + 2 * i], scale_log2, neg_m));
          const float p1 = ex2(fmaf(s[h * 32 + 2 * i + 1], scale_log2, neg_m));
          part[i & 3] += p0 + p1;
          pk[i] = pack2<BF16>(p0, p1);
        }
        tmem_st16(tmem_addr(tbase, lane_base, s_col + col0 / 2 + h * 16), pk);
      }
      const float sum = (part[0] + part[1]) + (part[2] + part[3]);
      if constexpr (R > 1) {
        // the other copies' key columns contribute nothing to this copy's rows
        const uint32_t zero[16] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
#pragma unroll
        for (int g = 0; g < BN / 32; ++g)
          if (g / (COLS / 32) != cp) tmem_st16(tmem_addr(tbase, lane_base, s_col + g * 16), zero);
      }
      l = l * alpha + sum;
      if (__any_sync(0xffffffffu, rescale)) {
        // O row *= alpha once P_{j-1} V_{j-1} has completed
        ok = __all_sync(0xffffffffu, mbar_wait(pv_done, (j - 1) & 1, ctx, 134));
        if (!ok) break;
        tc_fence_after();
        const float a = rescale ? alpha : 1.f;
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          uint32_t r[32];
          const uint32_t ta = tmem_addr(tbase, lane_base, C::O_COL + c * 32);
          tmem_ld32(ta, r);
          tmem_wait_ld();
          reg_fence(r);
#pragma unroll
          for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * a);
          tmem_st32(ta, r);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(p_full + (j & 1));
    }
    // ---------------------------------------------------------------- epilogue
    if (nb == 0) {
      // an empty piece (more pieces than key tiles): contributes nothing to the merge
      if (ok && cp == 0 && valid) {
        const int64_t grow = row_base + r0 + rit;
        float* wo = ws_o + (grow * splits + split) * D;
        for (int c = 0; c < D; c += 4) *reinterpret_cast<float4*>(wo + c) = make_float4(0.f, 0.f, 0.f, 0.f);
        ws_l[grow * splits + split] = -INFINITY;
      }
    } else if constexpr (R == 1) {
      if (warp_active && ok) ok = __all_sync(0xffffffffu, mbar_wait(o_full, 0, ctx, 140));
      if (warp_active && ok) {
        tc_fence_after();
        const int64_t grow = row_base + r0 + rit;  // row of Q, O, L ([B][H][Nq] flattened)
        const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          uint32_t r[32];
          tmem_ld32(tmem_addr(tbase, lane_base, C::O_COL + c * 32), r);
          tmem_wait_ld();
          reg_fence(r);
          if (valid && splits == 1) {
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
              pk[i] = pack2<BF16>(__uint_as_float(r[2 * i]) * inv, __uint_as_float(r[2 * i + 1]) * inv);
            uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(out) + (grow * D + c * 32) * 2);
#pragma unroll
            for (int i = 0; i < 4; ++i) dst[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
          } else if (valid) {
            float4* dst = reinterpret_cast<float4*>(ws_o + (grow * splits + split) * D + c * 32);
#pragma unroll
            for (int i = 0; i < 8; ++i)
              dst[i] = make_float4(__uint_as_float(r[4 * i]) * inv, __uint_as_float(r[4 * i + 1]) * inv,
                                   __uint_as_float(r[4 * i + 2]) * inv, __uint_as_float(r[4 * i + 3]) * inv);
          }
        }
        if (valid) {
          const float lse2 = l > 0.f ? m + log2f(l) : -INFINITY;
          if (splits == 1)
            lse[grow] = lse2 * 0.6931471805599453f;
          else
            ws_l[grow * splits + split] = lse2;
        }
        if (counter && warp == 0 && lane == 0) atomicAdd(counter, (unsigned long long)nb);
      }
    } else {
      // R copies of each row: merge them in shared memory (the ring is idle once o_full has
      // completed: every MMA is done and every load was consumed).  All four warps pass both
      // named barriers whatever happened before, so none can be left waiting.
      float* st_m = reinterpret_cast<float*>(smem + C::OFF_RING);  // [R][QR]
      float* st_l = st_m + BM;                                     // [R][QR]
      float* ob = st_l + BM;                                       // [R][QR][OROW]
      const int slot = cp * QR + rit;
      const bool mine = ok && __all_sync(0xffffffffu, mbar_wait(o_full, 0, ctx, 140));
      if (mine) {
        tc_fence_after();
        st_m[slot] = m;
        st_l[slot] = l;
      }
      named_bar_sync(kMergeBarrier, 128);
      // this row's combined maximum and sum; this copy's weight 2^(m - M) / l_total
      auto row_stats = [&](int r, float* mtot, float* ltot) {
        float mm = -INFINITY, ll = 0.f;
#pragma unroll
        for (int k = 0; k < R; ++k) mm = fmaxf(mm, st_m[k * QR + r]);
#pragma unroll
        for (int k = 0; k < R; ++k) {
          const float mk = st_m[k * QR + r];
          if (mk != -INFINITY) ll = fmaf(st_l[k * QR + r], ex2(mk - mm), ll);
        }
        *mtot = mm;
        *ltot = ll;
      };
      if (mine) {
        float mm, ll;
        row_stats(rit, &mm, &ll);
        const float f = (m == -INFINITY || !(ll > 0.f)) ? 0.f : ex2(m - mm) / ll;
        float* orow = ob + slot * C::OROW;
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          uint32_t r[32];
          tmem_ld32(tmem_addr(tbase, lane_base, C::O_COL + c * 32), r);
          tmem_wait_ld();
          reg_fence(r);
#pragma unroll
          for (int i = 0; i < 8; ++i)
            *reinterpret_cast<float4*>(orow + c * 32 + 4 * i) =
                make_float4(__uint_as_float(r[4 * i]) * f, __uint_as_float(r[4 * i + 1]) * f,
                            __uint_as_float(r[4 * i + 2]) * f, __uint_as_float(r[4 * i + 3]) * f);
        }
      }
      named_bar_sync(kMergeBarrier, 128);
      if (mine) {
        // the tile's rows, D / 4 four-element groups each, stored by the 128 threads together
        const int tid = threadIdx.x;
        for (int e = tid; e < mc * (D / 4); e += 128) {
          const int r = e / (D / 4), c4 = e - r * (D / 4);
          float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
          for (int k = 0; k < R; ++k) {
            const float4 v = *reinterpret_cast<const float4*>(ob + (k * QR + r) * C::OROW + c4 * 4);
            acc.x += v.x;
            acc.y += v.y;
            acc.z += v.z;
            acc.w += v.w;
          }
          const int64_t grow = row_base + r0 + r;
          if (splits == 1) {
            uint2* dst = reinterpret_cast<uint2*>(reinterpret_cast<uint8_t*>(out) + (grow * D + c4 * 4) * 2);
            *dst = make_uint2(pack2<BF16>(acc.x, acc.y), pack2<BF16>(acc.z, acc.w));
          } else {
            *reinterpret_cast<float4*>(ws_o + (grow * splits + split) * D + c4 * 4) = acc;
          }
        }
        if (tid < mc) {
          float mm, ll;
          row_stats(tid, &mm, &ll);
          const float lse2 = ll > 0.f ? mm + log2f(ll) : -INFINITY;
          const int64_t grow = row_base + r0 + tid;
          if (splits == 1)
            lse[grow] = lse2 * 0.6931471805599453f;
          else
            ws_l[grow * splits + split] = lse2;
        }
        if (counter && tid == 0) atomicAdd(counter, (unsigned long long)nb);
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

// copies of the tile's rows spread over the four lane quarters (see the top of the file)
int row_copies(int d, int rows) {
  if (d == 256) return 1;
  return rows <= 32 ? 4 : (rows <= 64 ? 2 : 1);
}

template <int D, bool BF16, int R>
cudaError_t launch_decode_tc_r(const DecodeArgs& a, const CUtensorMap& tk, const CUtensorMap& tv) {
  using C = DecCfg<D>;
  const int rows = (a.h / a.hkv) * a.nq;
  const int row_tiles = (rows + BM - 1) / BM;
  auto kern = decode_tc_kernel<D, BF16, R>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  const int64_t ctas = (int64_t)a.b * a.hkv * row_tiles * a.splits;
  const int64_t nrows = (int64_t)a.b * a.h * a.nq;
  float* ws_o = a.splits > 1 ? a.ws : nullptr;
  float* ws_l = a.splits > 1 ? a.ws + nrows * a.splits * D : nullptr;
  kern<<<(unsigned)ctas, C::THREADS, C::SMEM, a.stream>>>(static_cast<const uint32_t*>(a.q), tk, tv, a.o, a.lse, ws_o, ws_l, rows, a.h * a.nq,
                                                          a.hkv, row_tiles, a.splits, a.nk,
                                                          a.scale * 1.4426950408889634f, a.err, a.counter);
  if ((e = cudaGetLastError()) != cudaSuccess || a.splits == 1) return e;
  return launch_decode_merge(a);
}

template <int D, bool BF16>
cudaError_t launch_decode_tc_d(const DecodeArgs& a) {
  using C = DecCfg<D>;
  CUtensorMap tk, tv;
  if (!make_tmap_16bit_3d(&tk, a.k, BF16, D, a.nk, (uint64_t)a.b * a.hkv, C::BN) ||
      !make_tmap_16bit_3d(&tv, a.v, BF16, D, a.nk, (uint64_t)a.b * a.hkv, C::BN))
    return cudaErrorInvalidValue;
  if constexpr (D == 256) {
    return launch_decode_tc_r<D, BF16, 1>(a, tk, tv);
  } else {
    switch (row_copies(D, (a.h / a.hkv) * a.nq)) {
      case 4: return launch_decode_tc_r<D, BF16, 4>(a, tk, tv);
      case 2: return launch_decode_tc_r<D, BF16, 2>(a, tk, tv);
      default: return launch_decode_tc_r<D, BF16, 1>(a, tk, tv);
    }
  }
}

}  // namespace

bool decode_tc_supported(int dtype, int d, int64_t q_rows) {
  // the Q tensor map addresses rows with 32-bit coordinates
  return (dtype == DT_BF16 || dtype == DT_FP16) && (d == 64 || d == 128 || d == 256) && q_rows < (1ll << 31);
}

int decode_tc_auto_splits(int b, int h, int hkv, int nq, int nk, int d) {
  // One CTA per SM (each holds all 512 TMEM columns).  Time model, per wave of up to kSmCount
  // CTAs: tiles per piece x max(a CTA's own time per tile, the wave's share of HBM per tile),
  // plus a fixed cost per wave and one for the merge pass.  A CTA alone streams about 65, 88
  // and 76 GB/s at d = 64, 128, 256 and the cache reads at about 7 TB/s (measured on GB300),
  // so about 100 CTAs already saturate HBM and a single full wave usually wins.
  const double bn = (d == 256) ? 64 : 128;
  const double tile_bytes = 2.0 * bn * d * 2;
  const double cta_rate = (d == 64) ? 65e9 : (d == 128 ? 88e9 : 76e9);
  const double hbm_rate = 7.0e12, wave_cost = 3e-6, merge_cost = 3e-6;
  const int64_t row_tiles = ((int64_t)(h / hkv) * nq + BM - 1) / BM;
  const int64_t base = (int64_t)b * hkv * row_tiles;
  const int64_t tiles = (nk + (int64_t)bn - 1) / (int64_t)bn;
  const int64_t cap = std::min<int64_t>(tiles, 256);
  int64_t best = 1;
  double best_time = 1e30;
  for (int64_t s = 1; s <= cap; ++s) {
    const int64_t per = (tiles + s - 1) / s;
    double time = s > 1 ? merge_cost : 0.0;
    for (int64_t left = base * s; left > 0; left -= kSmCount) {
      const double n = (double)std::min<int64_t>(left, kSmCount);
      time += per * std::max(tile_bytes / cta_rate, n * tile_bytes / hbm_rate) + wave_cost;
    }
    if (time < best_time * 0.999) {
      best_time = time;
      best = s;
    }
  }
  return (int)best;
}

cudaError_t launch_decode_tc(const DecodeArgs& a) {
  const bool bf = a.dtype == DT_BF16;
  switch (a.d) {
    case 64: return bf ? launch_decode_tc_d<64, true>(a) : launch_decode_tc_d<64, false>(a);
    case 128: return bf ? launch_decode_tc_d<128, true>(a) : launch_decode_tc_d<128, false>(a);
    case 256: return bf ? launch_decode_tc_d<256, true>(a) : launch_decode_tc_d<256, false>(a);
    default: return cudaErrorNotSupported;
  }
}

}  // namespace fa
