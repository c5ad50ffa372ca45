// Tensor-core forward for bf16/fp16, head dims 64/128/256 (sm_103a: TMA, tcgen05, TMEM).
//
// What it computes (per head, rows i of Q): O_i = softmax(tau q_i K^T [+ causal mask]) V and
// L_i = m_i + ln l_i, exactly, with S and P only ever on chip ("Lecture 8 · GPU Performance
// & FlashAttention" §5.3 tiled forward, §5.4 what is kept for the backward; "FlashAttention
// and GPU memory" §07/§08).
//
// Work split (FA2 order, "Lecture 8" §8.1): a work item is NQ query tiles of 128 rows of one
// head; the CTA working on it streams 128-key tiles K_j, V_j through a shared-memory ring.
// Roles:
//   * softmax warpgroup q (4 warps, one thread per query row): reads S_q from TMEM,
//     applies the causal/ragged mask, runs the online softmax in the exp2 domain (§5.2),
//     writes P (16-bit) back into TMEM over S, rescales the O accumulator in TMEM when the
//     running maximum grows, and at the end divides by l and stores O and L;
//   * TMA warp: Q once, then K_j and V_j into the ring (rows past N read as zeros);
//   * MMA warp (one thread): S_q = Q_q K_j^T (both operands in smem) and
//     O_q += P_q V_j (P from TMEM, V from smem), accumulating in TMEM.
// With NQ = 2 (d = 64, 128) the two query tiles ping-pong: while one warpgroup does its
// softmax the tensor core runs the other tile's GEMMs (the interleave of "FlashAttention
// and GPU memory" §11).  With NQ = 1 (d = 256: O alone fills half of TMEM) S is
// double-buffered instead, so S_{j+1} is computed during the softmax of block j; the ring then
// holds 64-column blocks of the tiles, in the order the tensor core uses them (K0 K1 V0 K2 V1
// ...), so that K_{j+2} streams in while P_j V_j runs.
//
// Lazy rescaling: the reference maximum m used in exp2(x - m) is only raised when the new
// block maximum exceeds it by more than 8 (log2 units); until then P <= 2^8.  The final
// O / l and L = m + ln l use the same m, so the result is unchanged (the online-softmax
// identity holds for any reference value, §5.2).
//
// Causal: key tiles wholly in the future of a query tile are never loaded or multiplied
// (§5.3 closing paragraph); only diagonal tiles are masked element-wise.
//
// Persistent: a CTA (one per SM) walks work items (head, NQ query tiles).  It takes them from
// a queue (a ticket counter drawn by the producer warp and published to the other roles) when
// the launch has a counter slot, else round by round across the grid: in grid order, or for
// causal launches whose items a host-side estimate balances better that way, backwards in odd
// rounds (heavy and light items pair up).  The K/V ring, S/P and O barriers keep their phases
// across items; q_empty (all of an item's S = Q K^T issued and done) lets the next item's Q
// load while the item finishes, and o_empty (the softmax has read O) lets the next item's first
// P V overwrite O, so one item's epilogue overlaps the next item's loads and first S tiles.
#include <cuda.h>
#include <cuda_runtime.h>
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <mutex>
#include <vector>

#include "kernels.h"
#include "ptx.cuh"
#include "tmap.h"

namespace fa {
namespace {

constexpr int BM = 128;  // query rows per tile
constexpr int BN = 128;  // keys per tile
constexpr float kRescaleThreshold = 8.0f;

// F8: the FP8 variant (E4M3 codes of Q, K, V with one scale per 128-row block, kind::f8f6f4
// MMAs).  Everything is laid out by bytes: a tile row is D * EB bytes, held in 128-byte column
// blocks with the 128-byte swizzle (64-byte rows, FP8 at d = 64, with the 64-byte swizzle), and
// an MMA k-step reads 32 bytes of a row (16 16-bit or 32 8-bit elements).
template <int D, bool F8 = false>
struct FwdCfg {
  static constexpr int EB = F8 ? 1 : 2;               // bytes per element of Q, K, V
  static constexpr int ROW = D * EB;                  // bytes per tile row
  static constexpr int SW = ROW < 128 ? ROW : 128;    // swizzle width (bytes)
  static constexpr int KB = ROW / SW;                 // column blocks per row
  static constexpr int BLK_COLS = SW / EB;            // elements per column block
  static constexpr int NQ = (D == 256) ? 1 : 2;
  static constexpr int Q_BYTES = BM * ROW;
  static constexpr int TILE_BYTES = BN * ROW;
  // ring entries: a whole K or V tile at d = 64, 128; at d = 256 one 128-byte column block of a
  // tile (16 KB), so that the blocks of K are released one by one as their MMAs finish.  The
  // 16-bit d = 256 ring holds two tiles (8 entries; 10 entries, with the tiles that wrap round
  // the end split into N = 128 halves, ran 4-7 % slower)
  static constexpr int RB = (D == 256) ? KB : 1;  // ring entries per tile
  static constexpr int ENTRY_BYTES = TILE_BYTES / RB;
  static constexpr int STAGES = F8 ? (D == 64 ? 16 : 8) : ((D == 64) ? 8 : (D == 128 ? 4 : 8));
  static constexpr int SOFTMAX_WARPS = 4 * NQ;
  static constexpr int PRODUCER_WARP = SOFTMAX_WARPS;
  static constexpr int MMA_WARP = SOFTMAX_WARPS + 1;
  static constexpr int THREADS = 32 * (SOFTMAX_WARPS + 2);
  // an MMA k-step: 32 bytes of a row; P V: the keys of one k-step of packed P (8 TMEM columns)
  static constexpr int QK_STEPS = ROW / 32;
  static constexpr int PV_KEYS = 32 / EB;
  static constexpr int P_COLS = BN / (4 / EB);  // TMEM columns of a packed P row (64 or 32)
  // TMEM columns
  static constexpr int S_COL0 = 0, S_COL1 = 128;
  static constexpr int O_COL0 = 256;
  static constexpr int O_COL1 = (NQ == 2) ? 256 + D : 256;
  // d = 64: P gets columns of its own (S, O and P of both query tiles fit in the 512), so the
  // next S = Q K^T may overwrite S as soon as the softmax has read it, before P V has run
  static constexpr bool SEP_P = (D == 64);
  static constexpr int P_COL0 = 256 + 2 * D, P_COL1 = 256 + 2 * D + P_COLS;
  static_assert(!SEP_P || P_COL1 + P_COLS <= 512, "TMEM columns");
  // shared memory
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_RING = NQ * Q_BYTES;
  static constexpr int OFF_BAR = OFF_RING + STAGES * ENTRY_BYTES;
  static constexpr int NBAR = 1 + 2 * STAGES + 2 + 2 + 2 + 2 + 3 + 4 + 4 + 4;
  // after the barriers: TMEM base, abort flag, the two work-item slots
  static constexpr int SMEM = OFF_BAR + NBAR * 8 + 32;
  // masked variant: the CTA's key-tile list after the barriers (4 ints, then uint16 tile
  // indices and uint8 visibility flags, nb rounded up to 16 entries each)
  static constexpr int OFF_LIST = SMEM;
  static constexpr int list_bytes(int nb) { return 16 + 3 * ((nb + 15) & ~15); }
  // unmasked variant: after the barriers, one epilogue staging box per softmax warpgroup
  // ([128 rows][64 columns] 16-bit, 128-byte swizzle, the layout of the O tensor map's box),
  // through which O leaves by TMA stores 64 columns at a time
  static constexpr int OFF_STG = (SMEM + 1023) & ~1023;
  static constexpr int STG_BOX = BM * 128;
  static constexpr int SMEM_STG = OFF_STG + NQ * STG_BOX;
};

struct FwdSmemBars {
  uint64_t* q_full;
  uint64_t* kv_full;
  uint64_t* kv_empty;
  uint64_t* s_full;   // [2]
  uint64_t* p_full;   // [2]
  uint64_t* o_full;   // [2]
  uint64_t* pv_done;  // [1] (NQ = 1)
  uint64_t* drain;    // [1]
  uint64_t* o_empty;  // [2] the softmax has read O_q of its last item
  uint64_t* q_empty;  // [1] every S = Q K^T of the last item is done (Q may be overwritten)
  uint64_t* item_full;   // [2] the producer published a work item in this slot (queue mode)
  uint64_t* item_empty;  // [2] every consumer warp has read it
  uint64_t* stg_free;    // [2] the last TMA store from softmax warpgroup q's staging box has read it
  uint64_t* stg_full;    // [2] every thread of warpgroup q has written its row into the box
  uint64_t* s_free;      // [2] (separate P) the softmax has read S_q: the next S_q may be computed
  uint64_t* pv_q;        // [2] (separate P) P_q V of the last tile is done: P_q and O_q are free
};

// Masked variant (block mask and/or window, "Lecture 8" §5.7 block-sparse attention): one warp
// lists, before the roles start, the key tiles that either query tile of the CTA can see (a
// tile is skipped when its block-mask byte is 0 or the causal/window bounds leave no visible
// score in it) with a flag per query tile; the producer, the MMA warp and the softmax walk
// that list.  A query tile processes every listed tile up to its own last visible one, the
// ones it cannot see fully masked, so both tiles keep the same ping-pong schedule.
// FP8 variant (F8): Q, K, V are E4M3 codes with one fp32 scale per 128-row block of each head
// ("Lecture 8" §8.1, "FlashAttention and GPU memory" §11); the scales enter the softmax as
//   S_ij = tau sq(i) sk(j) (Q8 K8^T)_ij      (one score factor per pair of tiles),
//   O_i  = sum_j P_ij sv(j) V8_j / l_i,
// with sv(j) folded into P before it is rounded to E4M3: P8 = E4M3(exp2(S st + log2 sv(j) - m)),
// where the running maximum m is taken over S st + log2 sv(j) itself, so P8 <= 2^8 (the
// lazy-rescale bound) and a row's largest weighted probabilities stay near 1, whatever the
// spread of the V scales.  l sums exp2(S st - m) (each tile's sum of P8's unrounded values
// divided by sv(j)), so O = (sum P8 V8) / l and L = (m + log2 l) ln 2 as in the 16-bit kernel.
struct F8Scales {
  const float* q = nullptr;  // [bh][nb]
  const float* k = nullptr;  // [bh / group][nb]
  const float* v = nullptr;  // [bh / group][nb]
};

template <int D, bool BF16, bool MASKED, bool QUEUE, bool F8 = false>
__global__ void __launch_bounds__(FwdCfg<D, F8>::THREADS, 1)
    fwd_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o, void* __restrict__ out, float* __restrict__ lse, int n,
                  int bh_count, int tiles_per_head, float scale_log2, int causal, int group, unsigned long long* err,
                  unsigned long long* counter, int window, const uint8_t* __restrict__ block_mask, int mask_heads,
                  int heads, int snake, unsigned* __restrict__ sched, int hgroup, F8Scales f8s) {
  using C = FwdCfg<D, F8>;
  static_assert(!(F8 && MASKED), "the FP8 variant has no masks");
  extern __shared__ __align__(1024) uint8_t smem[];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  FwdSmemBars B;
  B.q_full = bars;
  B.kv_full = bars + 1;
  B.kv_empty = bars + 1 + C::STAGES;
  B.s_full = bars + 1 + 2 * C::STAGES;
  B.p_full = B.s_full + 2;
  B.o_full = B.p_full + 2;
  B.pv_done = B.o_full + 2;
  B.drain = B.pv_done + 1;
  B.o_empty = B.drain + 1;
  B.q_empty = B.o_empty + 2;
  B.item_full = B.q_empty + 1;
  B.item_empty = B.item_full + 2;
  B.stg_free = B.item_empty + 2;
  B.stg_full = B.stg_free + 2;
  B.s_free = B.stg_full + 2;
  B.pv_q = B.s_free + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::NBAR);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* item_slot = reinterpret_cast<volatile int*>(tmem_slot + 2);  // [2]
  // queue mode: items come from a ticket counter (sched) through the producer (never masked)
  constexpr bool queue = QUEUE && !MASKED;
  const ErrCtx ctx{err, abort_flag};

  // work items: head-major (CTAs running together share K/V in L2); causal: heaviest (last)
  // query tiles first within groups of heads
  const int total_items = bh_count * tiles_per_head;
  const int nblocks = (n + BN - 1) / BN;
  struct Item {
    int head, kvhead, qrow0;
    int nq[2];  // key tiles of each query tile
  };
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
    w.kvhead = w.head / group;  // grouped-query attention: key/value head shared by `group` query heads
    w.qrow0 = tile * (C::NQ * BM);
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const int first = w.qrow0 + q * BM;
      if (q >= C::NQ || first >= n) {
        w.nq[q] = 0;
      } else if (causal) {
        w.nq[q] = min(nblocks, (min(first + BM, n) - 1) / BN + 1);
      } else {
        w.nq[q] = nblocks;
      }
    }
    return w;
  };
  int* list_hdr = reinterpret_cast<int*>(smem + C::OFF_LIST);  // nq[0], nq[1], visible tiles of q 0, 1
  uint16_t* jlist = reinterpret_cast<uint16_t*>(smem + C::OFF_LIST + 16);
  uint8_t* jflag = reinterpret_cast<uint8_t*>(jlist + ((nblocks + 15) & ~15));
  if constexpr (MASKED) {
    if (warp == C::PRODUCER_WARP) {
      // (masked launches give every CTA one item, blockIdx.x)
      const int head = item_of(blockIdx.x).head, qrow0 = item_of(blockIdx.x).qrow0;
      // visible key tiles of query tile q: block-mask byte set, and some (row, key) pair of the
      // two tiles inside the causal and window bounds
      int qr0[2], qr1[2];
      const uint8_t* mrow[2] = {nullptr, nullptr};
      const int mh = mask_heads > 1 ? head % heads : 0;
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        qr0[q] = qrow0 + q * BM;
        qr1[q] = min(n, qr0[q] + BM) - 1;
        if (block_mask && q < C::NQ && qr0[q] < n)
          mrow[q] = block_mask + ((int64_t)mh * nblocks + qr0[q] / BM) * nblocks;
      }
      auto visible = [&](int q, int j) {
        if (q >= C::NQ || qr0[q] >= n) return false;
        const int kmin = j * BN, kmax = min(n, kmin + BN) - 1;
        bool v = !block_mask || mrow[q][j] != 0;
        if (causal) v = v && kmin <= qr1[q];
        if (window > 0) {
          v = v && qr0[q] - kmax < window;
          if (!causal) v = v && kmin - qr1[q] < window;
        }
        return v;
      };
      int count = 0, last0 = -1, last1 = -1, nv0 = 0, nv1 = 0;
      for (int base = 0; base < nblocks; base += 32) {
        const int j = base + lane;
        const bool v0 = j < nblocks && visible(0, j);
        const bool v1 = j < nblocks && visible(1, j);
        const unsigned any = __ballot_sync(0xffffffffu, v0 || v1);
        const unsigned b0 = __ballot_sync(0xffffffffu, v0), b1 = __ballot_sync(0xffffffffu, v1);
        if (v0 || v1) {
          const int pos = count + __popc(any & ((1u << lane) - 1u));
          jlist[pos] = (uint16_t)j;
          jflag[pos] = (uint8_t)((v0 ? 1 : 0) | (v1 ? 2 : 0));
        }
        if (b0) last0 = count + __popc(any & ((1u << (31 - __clz(b0))) - 1u));
        if (b1) last1 = count + __popc(any & ((1u << (31 - __clz(b1))) - 1u));
        nv0 += __popc(b0);
        nv1 += __popc(b1);
        count += __popc(any);
      }
      if (lane == 0) {
        list_hdr[0] = last0 + 1;
        list_hdr[1] = last1 + 1;
        list_hdr[2] = nv0;
        list_hdr[3] = nv1;
      }
    }
  }

  if (threadIdx.x == 0) {
    if ((smem_u32(smem) & 1023u) != 0) report_error(err, DERR_BAD_SMEM_ALIGN, 0);
    *abort_flag = (smem_u32(smem) & 1023u) != 0;
    mbar_init(B.q_full, 1);
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(B.kv_full + s, 1);
      mbar_init(B.kv_empty + s, 1);
    }
    for (int q = 0; q < 2; ++q) {
      mbar_init(B.s_full + q, 1);
      mbar_init(B.p_full + q, 128);
      mbar_init(B.o_full + q, 1);
    }
    mbar_init(B.pv_done, 1);
    mbar_init(B.drain, 1);
    mbar_init(B.o_empty + 0, 128);
    mbar_init(B.o_empty + 1, 128);
    mbar_init(B.q_empty, 1);
    for (int t = 0; t < 2; ++t) {
      mbar_init(B.item_full + t, 1);
      mbar_init(B.item_empty + t, C::SOFTMAX_WARPS + 1);  // the softmax warps and the MMA warp
      mbar_init(B.stg_free + t, 1);
      mbar_init(B.stg_full + t, 128);
      mbar_init(B.s_free + t, 128);
      mbar_init(B.pv_q + t, 1);
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
  // this CTA's r-th item: rounds of gridDim.x items, in grid order, or (snake) backwards in odd
  // rounds so that a CTA's heavy and light causal items pair up; -1 when done.  The grid size and
  // CTA index are read afresh each time (volatile reads cannot be hoisted): kept live across the
  // softmax loop they cost the d = 128 kernel spills.
  auto nth_item = [&](int r) {
    const int g = (int)grid_dim_x(), c = (int)cta_id_x();
    const int64_t item = (int64_t)r * g + ((snake && (r & 1)) ? (g - 1 - c) : c);
    return item < total_items ? (int)item : -1;
  };
  // this CTA's r-th item for a consumer warp: queue mode reads the producer's slot r % 2 (every
  // consumer warp reads every slot once; `good` turns false, and the item -1, when the bounded
  // wait ran out), otherwise the static order above
  auto next_item = [&](int r, bool& good) {
    if constexpr (!queue) return nth_item(r);
    const int t = r & 1;
    good = __all_sync(0xffffffffu, mbar_wait(B.item_full + t, (uint32_t)(r >> 1) & 1, ctx, 50)) && good;
    const int item = good ? item_slot[t] : -1;
    __syncwarp();
    if (lane == 0) mbar_arrive(B.item_empty + t);
    return item;
  };
  // the item with, for masked launches, the key-tile counts of its list
  auto item_at = [&](int item) {
    Item w = item_of(item);
    if constexpr (MASKED) {
      w.nq[0] = list_hdr[0];
      w.nq[1] = list_hdr[1];
    }
    return w;
  };
  // key tile at position t of an item's sequence
  auto tile_at = [&](int t) { return MASKED ? (int)jlist[t] : t; };
  // order of an item's K and V tiles in the ring (n key tiles): K0 V0 K1 V1 ... with two query
  // tiles (both tiles' GEMMs use a pair in turn); with one (S double-buffered) the order in which
  // the tensor core uses them, K0 K1 V0 K2 V1 ... K(n-1) V(n-2) V(n-1), so that the ring is
  // released and refilled first in, first out
  auto ring_tile = [&](int idx, int n_, bool* is_v, int* j) {
    if constexpr (C::NQ == 2) {
      *is_v = idx & 1;
      *j = idx >> 1;
    } else if (idx == 0) {
      *is_v = false;
      *j = 0;
    } else if (idx == 2 * n_ - 1) {
      *is_v = true;
      *j = n_ - 1;
    } else {
      *is_v = !(idx & 1);
      *j = (idx & 1) ? (idx + 1) >> 1 : (idx - 2) >> 1;
    }
  };
  // ring positions of K_j and V_j within the item (the inverse of ring_tile)
  auto k_pos = [&](int j, int n_) { return C::NQ == 2 ? 2 * j : (j == 0 ? 0 : 2 * j - 1); };
  auto v_pos = [&](int j, int n_) { return C::NQ == 2 ? 2 * j + 1 : (j == n_ - 1 ? 2 * n_ - 1 : 2 * j + 2); };

  if (warp == C::PRODUCER_WARP) {
    // ------------------------------------------------------------------ TMA producer
    if (start_ok && lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      uint32_t ring_pos = 0;  // ring loads issued so far (all items)
      int q_loads = 0;
      bool ok = true;
      // the r-th item: queue mode draws a ticket (items are numbered heaviest first) and publishes
      // it, or -1 once the queue is empty, when every reader of the slot's previous item has it
      auto draw = [&](int r) {
        if constexpr (!queue) return nth_item(r);
        if (r >= 2 && !(ok = mbar_wait(B.item_empty + (r & 1), (uint32_t)((r - 2) >> 1) & 1, ctx, 14))) return -1;
        const unsigned ticket = atomicAdd(sched, 1u);
        const int item = ticket < (unsigned)total_items ? (int)ticket : -1;
        item_slot[r & 1] = item;
        mbar_arrive(B.item_full + (r & 1));
        return item;
      };
      for (int r = 0, item = draw(0); ok && item >= 0; item = draw(++r)) {
        const Item w = item_at(item);
        const int nmax = max(w.nq[0], w.nq[1]);
        if (!(ok = debug_check(w.head < bh_count && w.kvhead * group < bh_count && w.qrow0 < n && nmax <= nblocks,
                               ctx, 60)))
          break;
        // Q of this item once the previous item's S = Q K^T are done
        if (q_loads > 0 && !(ok = mbar_wait(B.q_empty, (q_loads - 1) & 1, ctx, 13))) break;
        mbar_arrive_expect_tx(B.q_full, C::NQ * C::Q_BYTES);
        for (int q = 0; q < C::NQ; ++q)
          for (int kb = 0; kb < C::KB; ++kb)
            tma_load_3d(smem + C::OFF_Q + q * C::Q_BYTES + kb * (BM * C::SW), &tm_q, B.q_full, kb * C::BLK_COLS,
                        w.qrow0 + q * BM, w.head);
        ++q_loads;
        for (int idx = 0; ok && idx < 2 * nmax; ++idx) {
          bool is_v;
          int j;
          ring_tile(idx, nmax, &is_v, &j);
          if (!(ok = debug_check(j >= 0 && j < nmax && tile_at(j) >= 0 && tile_at(j) < nblocks, ctx, 61))) break;
          const CUtensorMap* tm = is_v ? &tm_v : &tm_k;
          for (int e = 0; e < C::RB; ++e) {
            const uint32_t g = ring_pos;
            const int slot = g % C::STAGES, use = g / C::STAGES;
            if (use > 0 && !(ok = mbar_wait(B.kv_empty + slot, (use - 1) & 1, ctx, 10))) break;
            mbar_arrive_expect_tx(B.kv_full + slot, C::ENTRY_BYTES);
            uint8_t* dst = smem + C::OFF_RING + slot * C::ENTRY_BYTES;
            constexpr int kbs = C::KB / C::RB;  // column blocks per entry
            for (int kb = 0; kb < kbs; ++kb)
              tma_load_3d(dst + kb * (BN * C::SW), tm, B.kv_full + slot, (e * kbs + kb) * C::BLK_COLS, tile_at(j) * BN,
                          w.kvhead);
            ++ring_pos;
          }
        }
      }
      // drain: every copy this thread started must land before the CTA may exit
      ErrCtx nctx = ctx;
      int no_abort = 0;
      nctx.abort = &no_abort;
      if (q_loads > 0) mbar_wait(B.q_full, (q_loads - 1) & 1, nctx, 11);
      for (int g = (int)ring_pos - 1; g >= 0 && g >= (int)ring_pos - C::STAGES; --g)
        mbar_wait(B.kv_full + g % C::STAGES, (g / C::STAGES) & 1, nctx, 12);
    }
    __syncwarp();
  } else if (warp == C::MMA_WARP) {
    // ------------------------------------------------------------------ MMA issuer
    // The whole warp runs this converged, so descriptors are warp-uniform; one elected lane
    // issues every MMA and commit (a commit tracks the MMAs of its own lane).
    if (start_ok) {
      const bool leader = elect_one_sync();
      // (FP8: E4M3 is format code 0 in the A and B fields of kind::f8f6f4, the layout of kind::f16)
      const uint32_t idesc_qk = make_idesc_f16(BM, BN, BF16 && !F8, false, false);
      const uint32_t idesc_pv = make_idesc_f16(BM, D, BF16 && !F8, false, true);
      const uint32_t q_base = smem_u32(smem + C::OFF_Q);
      const uint32_t ring = smem_u32(smem + C::OFF_RING);
      uint32_t ring_pos = 0;    // ring entry of the item's first tile (all items so far)
      int tq[2] = {0, 0};       // key tiles processed by each query tile (all items): P phases
      int oq[2] = {0, 0};       // items with a result for each query tile: O phases
      int items = 0;
      // ring slot of entry e of the tile at position idx of the item
      auto slot_of = [&](int idx, int e = 0) { return (int)((ring_pos + idx * C::RB + e) % C::STAGES); };
      auto wait = [&](uint64_t* b, uint32_t parity, uint32_t site) {
        return __all_sync(0xffffffffu, mbar_wait(b, parity, ctx, site));
      };
      // every entry of the tile at position idx has landed
      auto wait_full = [&](int idx) {
        bool good = true;
#pragma unroll
        for (int e = 0; e < C::RB; ++e)
          good = good && wait(B.kv_full + slot_of(idx, e), ((ring_pos + idx * C::RB + e) / C::STAGES) & 1, 20);
        return good;
      };
      auto commit = [&](uint64_t* b) {
        if (leader) umma_commit(b);
        __syncwarp();
      };
      // shared-memory descriptors of the tile layout (128- or 64-byte swizzle) and the MMA kind
      auto sdesc = [](uint32_t addr, uint32_t lbo, uint32_t sbo) {
        if constexpr (C::SW == 128) return make_sdesc_sw128(addr, lbo, sbo);
        else return make_sdesc_sw64(addr, lbo, sbo);
      };
      auto mma_ss = [](uint32_t d, uint64_t a, uint64_t b, uint32_t id, uint32_t acc) {
        if constexpr (F8) umma_ss_f8(d, a, b, id, acc);
        else umma_ss(d, a, b, id, acc);
      };
      auto mma_ts = [](uint32_t d, uint32_t a, uint64_t b, uint32_t id, uint32_t acc) {
        if constexpr (F8) umma_ts_f8(d, a, b, id, acc);
        else umma_ts(d, a, b, id, acc);
      };
      // S = Q_q K^T into TMEM columns s_col.  With block entries (d = 256) each 64-column block
      // of K is released as soon as its four MMAs are done.
      auto issue_qk = [&](int q, int kidx, uint32_t s_col) {
        const uint32_t qt = q_base + q * C::Q_BYTES;
        if constexpr (C::RB == 1) {
          const uint32_t kt = ring + slot_of(kidx) * C::ENTRY_BYTES;
          uint64_t ad[C::QK_STEPS], bd[C::QK_STEPS];
#pragma unroll
          for (int kk = 0; kk < C::QK_STEPS; ++kk) {
            const int b0 = kk * 32;  // byte offset of the k-step in the row
            ad[kk] = sdesc(qt + (b0 / C::SW) * (BM * C::SW) + (b0 % C::SW), 16, 8 * C::SW);
            bd[kk] = sdesc(kt + (b0 / C::SW) * (BN * C::SW) + (b0 % C::SW), 16, 8 * C::SW);
          }
          if (leader) {
#pragma unroll
            for (int kk = 0; kk < C::QK_STEPS; ++kk) mma_ss(tbase + s_col, ad[kk], bd[kk], idesc_qk, kk > 0);
          }
          __syncwarp();
        } else {
#pragma unroll
          for (int e = 0; e < C::RB; ++e) {
            const int slot = slot_of(kidx, e);
            const uint32_t kt = ring + slot * C::ENTRY_BYTES;
            uint64_t ad[4], bd[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              ad[i] = make_sdesc_sw128(qt + e * (BM * 128) + i * 32, 16, 1024);
              bd[i] = make_sdesc_sw128(kt + i * 32, 16, 1024);
            }
            if (leader) {
#pragma unroll
              for (int i = 0; i < 4; ++i) mma_ss(tbase + s_col, ad[i], bd[i], idesc_qk, (e > 0 || i > 0) ? 1u : 0u);
              umma_commit(B.kv_empty + slot);
            }
            __syncwarp();
          }
        }
      };
      // O += P V with P (16-bit, packed pairs) in TMEM columns [p_col, p_col + 64).  With block
      // entries (d = 256) a tile starts at a multiple of its entries and the ring holds a whole
      // number of tiles, so the blocks of V are adjacent (one N = 256 MMA per 16 keys, as for a
      // whole tile); they are released together.
      auto issue_pv = [&](uint32_t o_col, uint32_t p_col, int vidx, bool acc) {
        if constexpr (C::RB == 1) {
          const uint32_t vt = ring + slot_of(vidx) * C::ENTRY_BYTES;
          uint64_t bd[BN / C::PV_KEYS];
#pragma unroll
          for (int kk = 0; kk < BN / C::PV_KEYS; ++kk) bd[kk] = sdesc(vt + kk * C::PV_KEYS * C::SW, BN * C::SW, 8 * C::SW);
          if (leader) {
#pragma unroll
            for (int kk = 0; kk < BN / C::PV_KEYS; ++kk)
              mma_ts(tbase + o_col, tbase + p_col + kk * 8, bd[kk], idesc_pv, (acc || kk > 0) ? 1u : 0u);
          }
          __syncwarp();
        } else {
          static_assert(C::STAGES % C::RB == 0, "a tile's blocks never wrap round the ring");
          const uint32_t vt = ring + slot_of(vidx, 0) * C::ENTRY_BYTES;
          uint64_t bd[BN / C::PV_KEYS];
#pragma unroll
          for (int kk = 0; kk < BN / C::PV_KEYS; ++kk) bd[kk] = sdesc(vt + kk * C::PV_KEYS * C::SW, C::ENTRY_BYTES, 8 * C::SW);
          if (leader) {
#pragma unroll
            for (int kk = 0; kk < BN / C::PV_KEYS; ++kk)
              mma_ts(tbase + o_col, tbase + p_col + kk * 8, bd[kk], idesc_pv, (acc || kk > 0) ? 1u : 0u);
#pragma unroll
            for (int e = 0; e < C::RB; ++e) umma_commit(B.kv_empty + slot_of(vidx, e));
          }
          __syncwarp();
        }
      };
      // the first P V of query tile q in an item overwrites O_q: the softmax must have read it
      auto o_free = [&](int q) { return oq[q] == 0 || wait(B.o_empty + q, (oq[q] - 1) & 1, 26 + q); };
      bool ok = true;
      for (int r = 0, item = next_item(0, ok); ok && item >= 0; item = next_item(++r, ok)) {
        const Item w = item_at(item);
        const int* nq = w.nq;
        const int nmax = max(nq[0], nq[1]);
        if (!(ok = wait(B.q_full, items & 1, 21))) break;
        tc_fence_after();
        if constexpr (C::NQ == 2) {
          if (nmax > 0) {
            if (!(ok = wait_full(0))) break;
            tc_fence_after();
            if (nq[0] > 0) { issue_qk(0, 0, C::S_COL0); commit(B.s_full + 0); }
            if (nq[1] > 0) { issue_qk(1, 0, C::S_COL1); commit(B.s_full + 1); }
            commit(B.kv_empty + slot_of(0));
          }
          if (nmax <= 1) commit(B.q_empty);  // every S of the item is issued
          if constexpr (C::SEP_P) {
            // S_q(j+1) goes out as soon as the softmax has read S_q(j) (s_free), P_q(j) V_j once
            // it has written P_q(j) (p_full); each P V tells the softmax (pv_q) that P_q and O_q
            // are free again.  In the order the events come: tile 0's S, tile 0's P V, tile 1's
            // S, tile 1's P V (query tile 1 runs half a period behind tile 0).
            for (int j = 0; ok && j < nmax; ++j) {
              const int vidx = 2 * j + 1, kidx = 2 * j + 2;
              const bool more = j + 1 < nmax;
              if (more && !(ok = wait_full(kidx))) break;
              if (j + 1 < nq[0]) {
                if (!(ok = wait(B.s_free + 0, (tq[0] + j) & 1, 28))) break;
                tc_fence_after();
                issue_qk(0, kidx, C::S_COL0);
                commit(B.s_full + 0);
              }
              if (!(ok = wait_full(vidx))) break;
              if (j < nq[0]) {
                if (!(ok = wait(B.p_full + 0, (tq[0] + j) & 1, 22))) break;
                if (j == 0 && !(ok = o_free(0))) break;
                tc_fence_after();
                issue_pv(C::O_COL0, C::P_COL0, vidx, j > 0);
                commit(B.pv_q + 0);
                if (j == nq[0] - 1) commit(B.o_full + 0);
              }
              if (j + 1 < nq[1]) {
                if (!(ok = wait(B.s_free + 1, (tq[1] + j) & 1, 29))) break;
                tc_fence_after();
                issue_qk(1, kidx, C::S_COL1);
                commit(B.s_full + 1);
              }
              if (more) commit(B.kv_empty + slot_of(kidx));  // both S_{j+1} issued
              if (j == nmax - 2) commit(B.q_empty);         // the item's last S are issued
              if (j < nq[1]) {
                if (!(ok = wait(B.p_full + 1, (tq[1] + j) & 1, 23))) break;
                if (j == 0 && !(ok = o_free(1))) break;
                tc_fence_after();
                issue_pv(C::O_COL1, C::P_COL1, vidx, j > 0);
                commit(B.pv_q + 1);
                if (j == nq[1] - 1) commit(B.o_full + 1);
              }
              commit(B.kv_empty + slot_of(vidx));
            }
          } else {
            for (int j = 0; ok && j < nmax; ++j) {
              const int vidx = 2 * j + 1, kidx = 2 * j + 2;
              if (!(ok = wait_full(vidx))) break;
              if (j < nq[0]) {
                if (!(ok = wait(B.p_full + 0, (tq[0] + j) & 1, 22))) break;
                if (j == 0 && !(ok = o_free(0))) break;
                tc_fence_after();
                issue_pv(C::O_COL0, C::S_COL0, vidx, j > 0);
                // O_0 is final: its epilogue need not wait for query tile 1's last P
                if (j == nq[0] - 1) commit(B.o_full + 0);
              }
              if (j + 1 < nmax) {
                if (!(ok = wait_full(kidx))) break;
                tc_fence_after();
              }
              if (j + 1 < nq[0]) { issue_qk(0, kidx, C::S_COL0); commit(B.s_full + 0); }
              if (j < nq[1]) {
                if (!(ok = wait(B.p_full + 1, (tq[1] + j) & 1, 23))) break;
                if (j == 0 && !(ok = o_free(1))) break;
                tc_fence_after();
                issue_pv(C::O_COL1, C::S_COL1, vidx, j > 0);
              }
              commit(B.kv_empty + slot_of(vidx));
              if (j + 1 < nq[1]) { issue_qk(1, kidx, C::S_COL1); commit(B.s_full + 1); }
              if (j + 1 < nmax) commit(B.kv_empty + slot_of(kidx));
              if (j == nmax - 2) commit(B.q_empty);  // the item's last S are issued
              if (j == nq[1] - 1) commit(B.o_full + 1);
            }
          }
        } else {
          // NQ == 1: S double-buffered in columns 0 / 128 (by the global tile count), O at 256
          const int nb = nq[0];
          auto buf = [&](int j) { return ((tq[0] + j) & 1) ? C::S_COL1 : C::S_COL0; };
          for (int j = 0; ok && j < 2 && j < nb; ++j) {
            if (!(ok = wait_full(k_pos(j, nb)))) break;
            tc_fence_after();
            issue_qk(0, k_pos(j, nb), buf(j));  // releases K_j's ring entries
            commit(B.s_full + ((tq[0] + j) & 1));
          }
          if (ok && nb <= 2) commit(B.q_empty);
          for (int j = 0; ok && j < nb; ++j) {
            const int vidx = v_pos(j, nb);
            const int t = tq[0] + j;
            if (!(ok = wait_full(vidx))) break;
            if (!(ok = wait(B.p_full + (t & 1), (t >> 1) & 1, 24))) break;
            if (j == 0 && !(ok = o_free(0))) break;
            tc_fence_after();
            issue_pv(C::O_COL0, buf(j), vidx, j > 0);  // releases V_j's ring entries
            commit(B.pv_done);
            if (j + 2 < nb) {
              const int kidx = k_pos(j + 2, nb);
              if (!(ok = wait_full(kidx))) break;
              tc_fence_after();
              issue_qk(0, kidx, buf(j));  // in order after P_j V_j, which reads this buffer
              commit(B.s_full + (t & 1));
              if (j + 2 == nb - 1) commit(B.q_empty);
            }
            if (j == nb - 1) commit(B.o_full + 0);
          }
        }
        ring_pos += 2 * nmax * C::RB;
        for (int q = 0; q < 2; ++q) {
          tq[q] += nq[q];
          oq[q] += nq[q] > 0 ? 1 : 0;
        }
        ++items;
      }
      // drain: all MMAs complete before TMEM is released
      ErrCtx nctx = ctx;
      int no_abort = 0;
      nctx.abort = &no_abort;
      commit(B.drain);
      mbar_wait(B.drain, 0, nctx, 25);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------ softmax warpgroups
    const int q = warp >> 2;
    const int quarter = warp & 3;
    const uint32_t lane_base = quarter * 32;
    const int rit = quarter * 32 + lane;
    const uint32_t o_col = q ? C::O_COL1 : C::O_COL0;
    int tq = 0;  // key tiles this query tile processed (all items): S / P phases
    int oq = 0;  // items with a result: O phases
    uint32_t stg_uses = 0;  // TMA stores from this warpgroup's staging box (all items)
    bool ok = start_ok;
    for (int r = 0, item = next_item(0, ok); ok && item >= 0; item = next_item(++r, ok)) {
      const Item w = item_at(item);
      const int head = w.head;
      const int row = w.qrow0 + q * BM + rit;
      const int nb = w.nq[q];
      float m = -INFINITY;  // reference maximum, log2 units (scores * tau * log2 e)
      float l = 0.f;
      // FP8: the query block's scale, and the key and value scales of the next key tile
      const int nblk_s = (n + BN - 1) / BN;
      float sq_log2 = scale_log2, sk_next = 1.f, sv_next = 1.f;
      if constexpr (F8) {
        const int qblk = min((w.qrow0 + q * BM) / BM, nblk_s - 1);
        sq_log2 = scale_log2 * f8s.q[(int64_t)head * nblk_s + qblk];
        if (nb > 0) {
          sk_next = f8s.k[(int64_t)w.kvhead * nblk_s];
          sv_next = f8s.v[(int64_t)w.kvhead * nblk_s];
        }
      }
      for (int j = 0; ok && j < nb; ++j) {
        const int t = tq + j;
        // score scale (log2 units per unit of S) and, FP8, log2 of the key tile's V scale,
        // which rides in P's exponent
        float st = scale_log2, pv = 1.f, lpv = 0.f;
        if constexpr (F8) {
          st = sq_log2 * sk_next;
          pv = sv_next;
          lpv = __log2f(pv);
          if (j + 1 < nb) {
            sk_next = f8s.k[(int64_t)w.kvhead * nblk_s + j + 1];
            sv_next = f8s.v[(int64_t)w.kvhead * nblk_s + j + 1];
          }
        }
        uint32_t s_col;
        uint64_t* sbar;
        uint32_t sparity;
        if constexpr (C::NQ == 2) {
          s_col = q ? C::S_COL1 : C::S_COL0;
          sbar = B.s_full + q;
          sparity = t & 1;
        } else {
          s_col = (t & 1) ? C::S_COL1 : C::S_COL0;
          sbar = B.s_full + (t & 1);
          sparity = (t >> 1) & 1;
        }
        ok = __all_sync(0xffffffffu, mbar_wait(sbar, sparity, ctx, 30 + q));
        if (!ok) break;
        tc_fence_after();
        // whole S row: all TMEM loads in flight before one wait
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
        if constexpr (C::SEP_P) {  // S_q is in registers: the next S_q may be computed over it
          tc_fence_before();
          mbar_arrive(B.s_free + q);
        }
        // visible columns [lo, hi) of this row: keys before N, (causal) not after the row,
        // (window) within the window; none when the tile is listed only for the other query tile
        const int jt = tile_at(j);
        int lo = 0, hi = n - jt * BN;
        if (causal) hi = min(hi, row - jt * BN + 1);
        if constexpr (MASKED) {
          if (window > 0) {
            lo = row - window + 1 - jt * BN;
            if (!causal) hi = min(hi, row + window - jt * BN);
          }
          if (!((jflag[j] >> q) & 1)) hi = lo = 0;
        }
        if (lo > 0 || hi < BN) {
#pragma unroll
          for (int c = 0; c < BN; ++c)
            if (c < lo || c >= hi) s[c] = -INFINITY;
        }
        const float mx = row_max3(s);
        const float m_blk = F8 ? mx * st + lpv : mx * st;
        float alpha = 1.f;
        bool rescale = false;
        if (m == -INFINITY) {
          m = m_blk;  // first visible block of this row: O is written fresh (or is still zero)
          alpha = 0.f;
        } else if (m_blk > m + kRescaleThreshold) {
          alpha = ex2(m - m_blk);
          m = m_blk;
          rescale = true;
        }
        const float neg_m = F8 ? ((m == -INFINITY) ? 0.f : -m) + lpv : ((m == -INFINITY) ? 0.f : -m);
        if constexpr (C::SEP_P) {
          // P_q and O_q are free once the previous tile's P V is done
          if (t > 0) {
            ok = __all_sync(0xffffffffu, mbar_wait(B.pv_q + q, (t - 1) & 1, ctx, 36 + q));
            if (!ok) break;
            tc_fence_after();
          }
        }
        const uint32_t p_col = C::SEP_P ? (q ? C::P_COL1 : C::P_COL0) : s_col;
        // two partial sums of pairs (paired fp32 adds): no single long add chain
        float2 part[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
        if constexpr (!F8) {
#pragma unroll
          for (int h = 0; h < BN / 32; ++h) {
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float2 x = ffma2(make_float2(s[h * 32 + 2 * i], s[h * 32 + 2 * i + 1]), st, neg_m);
              const float2 pp = make_float2(ex2(x.x), ex2(x.y));
              part[i & 1] = fadd2(part[i & 1], pp);
              pk[i] = pack2<BF16>(pp.x, pp.y);
            }
            tmem_st16(tmem_addr(tbase, lane_base, p_col + h * 16), pk);
          }
        } else {
          // E4M3, four to a TMEM column
#pragma unroll
          for (int h = 0; h < BN / 64; ++h) {
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float* sv4 = &s[h * 64 + 4 * i];
              const float2 x01 = ffma2(make_float2(sv4[0], sv4[1]), st, neg_m);
              const float2 x23 = ffma2(make_float2(sv4[2], sv4[3]), st, neg_m);
              const float2 p01 = make_float2(ex2(x01.x), ex2(x01.y)), p23 = make_float2(ex2(x23.x), ex2(x23.y));
              part[i & 1] = fadd2(part[i & 1], fadd2(p01, p23));
              pk[i] = pack4_e4m3(p01.x, p01.y, p23.x, p23.y);
            }
            tmem_st16(tmem_addr(tbase, lane_base, p_col + h * 16), pk);
          }
        }
        // (FP8: the values carry sv; dividing their sum by it gives the sum of exp2(S st - m))
        const float sum = F8 ? ((part[0].x + part[1].x) + (part[0].y + part[1].y)) / pv
                             : (part[0].x + part[1].x) + (part[0].y + part[1].y);
        l = l * alpha + sum;
        if (__any_sync(0xffffffffu, rescale)) {
          // O row *= alpha; O is stable: the PV of block j-1 completed before S_j (NQ = 2 without
          // separate P: same issuing thread, in order), or pv_done (NQ = 1) / pv_q (separate P,
          // waited above) says so.
          if constexpr (C::NQ == 1) {
            ok = __all_sync(0xffffffffu, mbar_wait(B.pv_done, (t - 1) & 1, ctx, 34));
            if (!ok) break;
            tc_fence_after();
          }
          const float a = rescale ? alpha : 1.f;
#pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            uint32_t r[32];
            const uint32_t ta = tmem_addr(tbase, lane_base, o_col + c * 32);
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
        // NQ = 1: one barrier per S buffer; with a single one the softmax could finish blocks j
        // and j + 1 while the MMA warp still waits for V_j, and its parity wait on phase j would
        // then see phase j + 1
        mbar_arrive(B.p_full + (C::NQ == 2 ? q : (t & 1)));
      }
      // epilogue: O / l -> global (16-bit), L = (m + log2 l) ln 2
      if (ok && nb > 0) {
        ok = __all_sync(0xffffffffu, mbar_wait(B.o_full + q, oq & 1, ctx, 40 + q));
        if (ok && !MASKED) {
          // 64 columns at a time: TMEM -> registers (x 1/l) -> this warpgroup's staging box ->
          // one TMA store (rows past N are not written).  The box is taken once the previous
          // store from it has read it; O is released (o_empty) as soon as its last columns are in
          // registers, so the next item's first P V need not wait for the stores.
          tc_fence_after();
          const float inv = l > 0.f ? 1.f / l : 0.f;
          uint8_t* box = smem + C::OFF_STG + q * C::STG_BOX;
          const bool leader = (rit == 0);
#pragma unroll 1
          for (int pc = 0; pc < D / 64 && ok; ++pc) {
            if (leader) {
              bulk_wait_group_read<0>();
              mbar_arrive(B.stg_free + q);
            }
            ok = __all_sync(0xffffffffu, mbar_wait(B.stg_free + q, stg_uses & 1, ctx, 44 + q));
            if (!ok) break;
            uint8_t* rp = box + rit * 128;
#pragma unroll 1
            for (int h = 0; h < 2; ++h) {
              uint32_t r[32];
              tmem_ld32(tmem_addr(tbase, lane_base, o_col + pc * 64 + h * 32), r);
              tmem_wait_ld();
              reg_fence(r);
              if (pc == D / 64 - 1 && h == 1) {  // O is in registers: the next item may overwrite it
                tc_fence_before();
                mbar_arrive(B.o_empty + q);
              }
#pragma unroll
              for (int u = 0; u < 4; ++u) {
                const uint32_t* v = &r[u * 8];
                const uint4 pk = make_uint4(pack2<BF16>(__uint_as_float(v[0]) * inv, __uint_as_float(v[1]) * inv),
                                            pack2<BF16>(__uint_as_float(v[2]) * inv, __uint_as_float(v[3]) * inv),
                                            pack2<BF16>(__uint_as_float(v[4]) * inv, __uint_as_float(v[5]) * inv),
                                            pack2<BF16>(__uint_as_float(v[6]) * inv, __uint_as_float(v[7]) * inv));
                const uint32_t ch = (uint32_t)(h * 4 + u);
                *reinterpret_cast<uint4*>(rp + ((ch ^ (uint32_t)(rit & 7)) << 4)) = pk;
              }
            }
            fence_proxy_async_smem();
            mbar_arrive(B.stg_full + q);
            if (leader) {
              ok = mbar_wait(B.stg_full + q, stg_uses & 1, ctx, 46 + q);
              if (ok) {
                tma_store_3d(&tm_o, box, pc * 64, w.qrow0 + q * BM, head);
                bulk_commit_group();
              }
            }
            ++stg_uses;
          }
          ++oq;
          if (row < n) lse[(int64_t)head * n + row] = l > 0.f ? (m + log2f(l)) * 0.6931471805599453f : -INFINITY;
          if (counter && rit == 0) atomicAdd(counter, (unsigned long long)nb);
        } else if (ok) {
          // masked launches (one item per CTA): rows straight from registers to global memory
          tc_fence_after();
          const float inv = l > 0.f ? 1.f / l : 0.f;
          uint8_t* orow = reinterpret_cast<uint8_t*>(out) + (((int64_t)head * n + row) * D) * 2;
#pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            uint32_t r[32];
            tmem_ld32(tmem_addr(tbase, lane_base, o_col + c * 32), r);
            tmem_wait_ld();
            reg_fence(r);
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
              pk[i] = pack2<BF16>(__uint_as_float(r[2 * i]) * inv, __uint_as_float(r[2 * i + 1]) * inv);
            if (row < n) {
              uint4* dst = reinterpret_cast<uint4*>(orow + c * 64);
#pragma unroll
              for (int i = 0; i < 4; ++i) dst[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
            }
          }
          // every TMEM load of O is done (each chunk waited): the next item may overwrite it
          tc_fence_before();
          mbar_arrive(B.o_empty + q);
          ++oq;
          if (row < n) lse[(int64_t)head * n + row] = l > 0.f ? (m + log2f(l)) * 0.6931471805599453f : -INFINITY;
          if (counter && rit == 0) atomicAdd(counter, (unsigned long long)(MASKED ? list_hdr[2 + q] : nb));
        }
      } else if (MASKED && ok && nb == 0 && row < n) {
        // no listed key tile for this query tile: its rows see no key (O = 0, L = -inf)
        uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(out) + (((int64_t)head * n + row) * D) * 2);
#pragma unroll 1
        for (int c = 0; c < D / 8; ++c) dst[c] = make_uint4(0u, 0u, 0u, 0u);
        lse[(int64_t)head * n + row] = -INFINITY;
      }
      tq += nb;
    }
    if (!MASKED && rit == 0) bulk_wait_group<0>();  // this warpgroup's TMA stores have completed
  }

  tc_fence_before();
  __syncthreads();
  if (warp == C::MMA_WARP) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
  if (queue && threadIdx.x == 0) {  // (queue: a compile-time constant)
    // this CTA draws no more tickets; the last one to get here empties the queue for the next
    // launch that uses it (every CTA has drawn its last ticket by then)
    __threadfence();
    if (atomicAdd(sched + 1, 1u) == gridDim.x - 1) {
      atomicExch(sched, 0u);
      atomicExch(sched + 1, 0u);
    }
  }
}

// Largest per-CTA work (key tiles) of a persistent causal grid of g CTAs over the items, in grid
// order or snake order: the same item order and key-tile counts as the kernel.
int64_t max_cta_tiles(int bh, int tiles_per_head, int n, int nq_tiles, int g, bool snake, int hgroup) {
  std::vector<int64_t> load(g, 0);
  const int64_t total = (int64_t)bh * tiles_per_head;
  const int nblocks = (n + BN - 1) / BN;
  for (int64_t r = 0; r * g < total; ++r)
    for (int c = 0; c < g; ++c) {
      const int64_t item = r * g + ((snake && (r & 1)) ? (g - 1 - c) : c);
      if (item >= total) continue;
      int head, rank;
      grouped_work_item((int)item, bh, tiles_per_head, hgroup, &head, &rank);
      const int tile = tiles_per_head - 1 - rank;
      for (int q = 0; q < nq_tiles; ++q) {
        const int first = tile * nq_tiles * BM + q * BM;
        if (first < n) load[c] += std::min(nblocks, (std::min(first + BM, n) - 1) / BN + 1);
      }
    }
  return *std::max_element(load.begin(), load.end());
}

// Launch of the persistent forward (16-bit, or FP8 when f8 carries the block scales; then
// Q, K, V of `a` are E4M3 codes and BF16 is O's type).
template <int D, bool BF16, bool MASKED, bool F8 = false>
cudaError_t launch_fwd_d(const FwdArgs& a, F8Scales f8 = F8Scales()) {
  using C = FwdCfg<D, F8>;
  CUtensorMap tq, tk, tv, to;
  const int bh_kv = a.bh / a.group;
  bool maps;
  if constexpr (F8)
    maps = make_tmap_8bit_3d(&tq, a.q, D, a.n, a.bh, BM, C::SW) && make_tmap_8bit_3d(&tk, a.k, D, a.n, bh_kv, BN, C::SW) &&
           make_tmap_8bit_3d(&tv, a.v, D, a.n, bh_kv, BN, C::SW);
  else
    maps = make_tmap_16bit_3d(&tq, a.q, BF16, D, a.n, a.bh, BM) && make_tmap_16bit_3d(&tk, a.k, BF16, D, a.n, bh_kv, BN) &&
           make_tmap_16bit_3d(&tv, a.v, BF16, D, a.n, bh_kv, BN);
  if (!maps || !make_tmap_16bit_3d(&to, a.o, BF16, D, a.n, a.bh, BM)) return cudaErrorInvalidValue;
  const int nblocks = (a.n + BN - 1) / BN;
  const int smem = MASKED ? C::SMEM + C::list_bytes(nblocks) : C::SMEM_STG;
  if (smem > 232448) return cudaErrorInvalidValue;  // key-tile list too long for shared memory
  const int tiles = (a.n + C::NQ * BM - 1) / (C::NQ * BM);
  const float scale_log2 = a.scale * 1.4426950408889634f;
  // one CTA per SM walking the items; masked launches keep one item per CTA (its tile list
  // lives in shared memory)
  const int64_t items = (int64_t)a.bh * tiles;
  const int64_t grid = MASKED ? items : std::min<int64_t>(items, device_sm_count());
  // causal order: groups of query heads whose K, V (shared by `group` query heads) stay in L2
  const int hgroup = head_group_for_l2((int64_t)2 * a.n * C::ROW / a.group, kL2HeadBudgetFwd);
  const int snake = (!MASKED && a.causal && grid < items &&
                     max_cta_tiles(a.bh, tiles, a.n, C::NQ, (int)grid, true, hgroup) <
                         max_cta_tiles(a.bh, tiles, a.n, C::NQ, (int)grid, false, hgroup))
                        ? 1
                        : 0;
  // with more items than CTAs: the queue when a slot is free (CTAs that finish early take more
  // items, whatever the cause), else the static order
  QueueSlot qs;
  if (!MASKED && grid < items) qs = queue_slot_take(a.stream);
  auto kern = fwd_tc_kernel<D, BF16, MASKED, false, F8>;
  if constexpr (!MASKED) {
    if (qs.slot >= 0) kern = fwd_tc_kernel<D, BF16, false, true, F8>;
  }
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e == cudaSuccess) {
    kern<<<(unsigned)grid, C::THREADS, smem, a.stream>>>(tq, tk, tv, to, a.o, a.lse, a.n, a.bh, tiles, scale_log2,
                                                         a.causal, a.group, a.err, a.counter, a.window, a.block_mask,
                                                         a.mask_heads, a.heads, snake, qs.counters, hgroup, f8);
    e = cudaGetLastError();
  }
  return queue_slot_done(qs, e, a.stream);
}

template <int D, bool BF16>
cudaError_t launch_fwd_dm(const FwdArgs& a) {
  return a.masked() ? launch_fwd_d<D, BF16, true>(a) : launch_fwd_d<D, BF16, false>(a);
}

}  // namespace

namespace {

// Work-item queues of the persistent forwards (16-bit and FP8; the calls have no workspace): a
// few pairs of counters (next ticket, CTAs done) in device memory that the library owns.  A
// stream keeps the slot of its last launch (launches on one stream run one after the other, so
// that launch has finished, and its last CTA has set the counters back to zero, before the next
// one starts).  A stream without a slot takes one that no unfinished launch uses: the event
// recorded on the stream right after the slot's last launch has completed.  A stream being
// captured into a graph, or finding every slot busy, gets no slot and the static order instead.
constexpr int kQueueSlots = 32;
constexpr int kMaxQueueDevices = 64;
__device__ unsigned g_fwd_queue[kQueueSlots][2];

struct QueuePool {
  unsigned* base = nullptr;
  cudaEvent_t done[kQueueSlots] = {};
  bool used[kQueueSlots] = {};    // a launch was recorded on done[i]
  bool broken[kQueueSlots] = {};  // recording failed: never reused
  bool owned[kQueueSlots] = {};   // owner[i] holds the stream of the slot's last launch
  unsigned long long owner[kQueueSlots] = {};
  int next = 0;
};
QueuePool g_qpool[kMaxQueueDevices];
std::mutex g_qpool_mu;  // held from choosing a slot until its launch is recorded

// A free slot of the current device's pool (its index; *counters its device address), or -1.
int acquire_queue_slot(cudaStream_t stream, QueuePool** pool, unsigned** counters, int* device) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone) return -1;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxQueueDevices) return -1;
  *device = dev;
  // streams are told apart by their ids, which (unlike handles) are never reused
  unsigned long long sid = 0;
  if (cudaStreamGetId(stream, &sid) != cudaSuccess) {
    (void)cudaGetLastError();
    return -1;
  }
  QueuePool& p = g_qpool[dev];
  if (!p.base) {
    void* b = nullptr;
    if (cudaGetSymbolAddress(&b, g_fwd_queue) != cudaSuccess || !b) return -1;
    p.base = static_cast<unsigned*>(b);
  }
  // the stream's own slot: launches on one stream run one after the other, so the slot's last
  // launch has finished (and reset the counters) before this one starts
  for (int i = 0; i < kQueueSlots; ++i) {
    if (p.owned[i] && p.owner[i] == sid && !p.broken[i]) {
      *pool = &p;
      *counters = p.base + 2 * i;
      return i;
    }
  }
  // else a slot whose last launch (on any stream) has completed; it changes owner
  for (int t = 0; t < kQueueSlots; ++t) {
    const int i = (p.next + t) % kQueueSlots;
    if (p.broken[i]) continue;
    if (!p.done[i] && cudaEventCreateWithFlags(&p.done[i], cudaEventDisableTiming) != cudaSuccess) {
      p.done[i] = nullptr;
      return -1;
    }
    if (p.used[i]) {
      const cudaError_t q = cudaEventQuery(p.done[i]);
      if (q == cudaErrorNotReady) {
        if (cudaPeekAtLastError() == cudaErrorNotReady) (void)cudaGetLastError();
        continue;
      }
      if (q != cudaSuccess) return -1;
    }
    p.next = (i + 1) % kQueueSlots;
    p.owned[i] = true;
    p.owner[i] = sid;
    *pool = &p;
    *counters = p.base + 2 * i;
    return i;
  }
  return -1;
}

}  // namespace

QueueSlot queue_slot_take(cudaStream_t stream) {
  QueueSlot q;
  g_qpool_mu.lock();
  QueuePool* pool = nullptr;
  q.slot = acquire_queue_slot(stream, &pool, &q.counters, &q.device);
  if (q.slot < 0) {
    q.counters = nullptr;
    g_qpool_mu.unlock();
  }
  return q;
}

cudaError_t queue_slot_done(const QueueSlot& q, cudaError_t launch_status, cudaStream_t stream) {
  if (q.slot < 0) return launch_status;
  QueuePool& p = g_qpool[q.device];
  cudaError_t e = launch_status;
  if (e == cudaSuccess) {
    e = cudaEventRecord(p.done[q.slot], stream);
    if (e == cudaSuccess)
      p.used[q.slot] = true;
    else
      p.broken[q.slot] = true;  // the launch may still run: never hand this slot out again
  }
  g_qpool_mu.unlock();
  return e;
}

bool fwd_masked_fits(int n, int d) {
  const int nb = (n + BN - 1) / BN;
  if (nb > 65535) return false;
  const int base = d == 64 ? FwdCfg<64>::SMEM : (d == 128 ? FwdCfg<128>::SMEM : FwdCfg<256>::SMEM);
  return base + FwdCfg<64>::list_bytes(nb) <= 232448;
}

bool fwd_fp8_supported(int d) { return d == 64 || d == 128 || d == 256; }

cudaError_t launch_fwd_fp8(const Fp8FwdArgs& a) {
  FwdArgs f{a.q8, a.k8, a.v8, a.o, a.lse, a.bh, a.n, a.d, a.scale, a.causal, a.out_dtype, a.err, a.counter, a.stream};
  f.group = a.group;
  f.heads = a.bh;
  F8Scales sc;
  sc.q = a.q_scales;
  sc.k = a.k_scales;
  sc.v = a.v_scales;
  const bool bf = a.out_dtype == DT_BF16;
  switch (a.d) {
    case 64: return bf ? launch_fwd_d<64, true, false, true>(f, sc) : launch_fwd_d<64, false, false, true>(f, sc);
    case 128: return bf ? launch_fwd_d<128, true, false, true>(f, sc) : launch_fwd_d<128, false, false, true>(f, sc);
    case 256: return bf ? launch_fwd_d<256, true, false, true>(f, sc) : launch_fwd_d<256, false, false, true>(f, sc);
    default: return cudaErrorNotSupported;
  }
}

bool fwd_tc_supported(int dtype, int d) {
  return (dtype == DT_BF16 || dtype == DT_FP16) && (d == 64 || d == 128 || d == 256);
}

cudaError_t launch_fwd_tc(const FwdArgs& a) {
  const bool bf = a.dtype == DT_BF16;
  switch (a.d) {
    case 64: return bf ? launch_fwd_dm<64, true>(a) : launch_fwd_dm<64, false>(a);
    case 128: return bf ? launch_fwd_dm<128, true>(a) : launch_fwd_dm<128, false>(a);
    case 256: return bf ? launch_fwd_dm<256, true>(a) : launch_fwd_dm<256, false>(a);
    default: return cudaErrorNotSupported;
  }
}

}  // namespace fa
