// Internal launch interface between the C ABI (api.cu) and the kernel files.
#pragma once
#include <cuda_runtime.h>
#include <cstdint>

namespace fa {

enum Dtype : int { DT_BF16 = 0, DT_FP16 = 1, DT_FP32 = 2 };

// Rows of the padded per-head statistics and of the fp32 dQ accumulator.
inline int64_t padded_rows(int64_t n) { return (n + 127) / 128 * 128; }

struct FwdArgs {
  const void* q;
  const void* k;
  const void* v;
  void* o;
  float* lse;
  int bh;  // B*H (query heads)
  int n;
  int d;
  float scale;
  int causal;
  int dtype;
  unsigned long long* err;      // device error word
  unsigned long long* counter;  // device count of processed (query tile, key tile) pairs
  cudaStream_t stream;
  int group = 1;  // query heads per key/value head: K, V hold bh / group heads
  // masks beyond causal (0 / null: none): keys with |i - j| >= window are hidden, and the
  // 128 x 128 score blocks whose byte in block_mask [mask_heads][nb][nb] is 0 (mask_heads is 1
  // or the number of query heads `heads`; nb = ceil(n / 128))
  int window = 0;
  const uint8_t* block_mask = nullptr;
  int mask_heads = 0;
  int heads = 1;
  bool masked() const { return window > 0 || block_mask != nullptr; }
};

// Backward workspace, carved from one caller buffer of fa_bwd_workspace_size bytes:
//   delta  [bh][npad]     fp32  D_i = sum_k dO_ik O_ik (0 on padding rows)
//   lse2   [bh][npad]     fp32  -L_i * log2(e) (-inf on padding rows and rows with L = -inf)
//   dq_acc [bh][npad][d]  fp32  accumulated dS K (before the factor tau)
struct BwdArgs {
  const void* q;
  const void* k;
  const void* v;
  const void* o;
  const void* dout;
  const float* lse;
  void* dq;
  void* dk;
  void* dv;
  float* delta;
  float* lse2;
  float* dq_acc;
  unsigned* sched = nullptr;  // [2] work-item queue of the tensor-core backward: next ticket, CTAs done
  int bh;
  int n;
  int d;
  float scale;
  int causal;
  int dtype;
  unsigned long long* err;
  unsigned long long* counter;
  cudaStream_t stream;
  int group = 1;  // query heads per key/value head: K, V, dK, dV hold bh / group heads
  int window = 0;  // masks beyond causal, as in FwdArgs
  const uint8_t* block_mask = nullptr;
  int mask_heads = 0;
  int heads = 1;
  bool masked() const { return window > 0 || block_mask != nullptr; }
};

// Decode over a key/value cache: Q, O [b][h][nq][d], K, V [b][hkv][nk][d], L [b][h][nq].
struct DecodeArgs {
  const void* q;
  const void* k;
  const void* v;
  void* o;
  float* lse;
  float* ws;  // splits > 1: [b*h*nq][splits][d] split outputs, then [b*h*nq][splits] base-2 LSEs
  int b, h, hkv, nq, nk, d;
  float scale;
  int splits;
  int dtype;
  cudaStream_t stream;
  unsigned long long* err = nullptr;      // device error word (tensor-core path)
  unsigned long long* counter = nullptr;  // device count of processed (row tile, key tile) pairs
};
// Heads per group of the causal work-item order (grouped_work_item): as many heads as keep
// `bytes_per_head` (what a head's items stream: K and V in the forward; Q, dO, the dQ
// accumulator, L and D in the backward) within an L2 budget, at least 1 and at most
// kMaxHeadGroup.  Forward: about a third of the 129 MB L2, as Q and O stream through it once;
// with 67 MB of K/V in flight (four heads of 65536 keys at d = 64) the forward read K/V twice
// over from DRAM, with 34 MB (two heads) once.  Backward: 80 MB; at 40 MB the causal LM shape
// (4 MB a head) ran 3 % slower and the 65536-key shape read 5 % less, in the same time.
#ifndef FA_L2_HEAD_BUDGET_FWD_MB
#define FA_L2_HEAD_BUDGET_FWD_MB 40
#endif
#ifndef FA_L2_HEAD_BUDGET_BWD_MB
#define FA_L2_HEAD_BUDGET_BWD_MB 80
#endif
constexpr int64_t kL2HeadBudgetFwd = (int64_t)FA_L2_HEAD_BUDGET_FWD_MB << 20;
constexpr int64_t kL2HeadBudgetBwd = (int64_t)FA_L2_HEAD_BUDGET_BWD_MB << 20;
inline int head_group_for_l2(int64_t bytes_per_head, int64_t budget) {
  const int64_t g = bytes_per_head > 0 ? budget / bytes_per_head : 16;
  return (int)(g < 1 ? 1 : (g > 16 ? 16 : g));  // 16: kMaxHeadGroup
}
// Streaming multiprocessors of a GB300, for sizing grids.
constexpr int kSmCount = 152;
// Unique id of the CUDA context current on the calling thread (ids are never reused), or 0 when
// no context is current or the driver cannot say.
unsigned long long current_context_id();
// Streaming multiprocessors of the current device (cached per device; kSmCount if unknown).
int device_sm_count();
int decode_auto_splits(int b, int h, int hkv, int nq, int nk);
int decode_tc_auto_splits(int b, int h, int hkv, int nq, int nk, int d);
bool decode_tc_supported(int dtype, int d, int64_t q_rows);
size_t decode_workspace_bytes(int b, int h, int nq, int d, int splits);
cudaError_t launch_decode(const DecodeArgs& a);     // CUDA cores, any dtype
cudaError_t launch_decode_tc(const DecodeArgs& a);  // tensor cores, bf16/fp16
cudaError_t launch_decode_merge(const DecodeArgs& a);

// FP8 (E4M3) block quantisation: X [bh][n][d] (dtype) -> codes X8 [bh][n][d] (bytes) and one
// fp32 scale per 128-row block, scales [bh][ceil(n / 128)].
struct QuantArgs {
  const void* x;
  void* x8;
  float* scales;
  int bh, n, d, dtype;
  cudaStream_t stream;
  unsigned long long* err = nullptr;  // device error word (bounded waits of the streaming kernel)
};
cudaError_t launch_quantize_fp8(const QuantArgs& a);

// Work-item queue slots of the persistent forwards (a library-owned pool of counter pairs).
// queue_slot_take picks a slot that no unfinished launch uses (slot -1, counters null: none
// free, or the stream is being captured into a graph) and holds the pool's lock until
// queue_slot_done, which must follow the launch at once with its status: it records the slot's
// completion event on the stream and returns the launch status (or the recording error).
struct QueueSlot {
  int slot = -1;
  int device = 0;
  unsigned* counters = nullptr;
};
QueueSlot queue_slot_take(cudaStream_t stream);
cudaError_t queue_slot_done(const QueueSlot& q, cudaError_t launch_status, cudaStream_t stream);

// FP8 forward: Q8, K8, V8 [bh][n][d] E4M3 codes with block scales; O [bh][n][d] in out_dtype
// (bf16 or fp16), L [bh][n] fp32.
struct Fp8FwdArgs {
  const void* q8;
  const void* k8;
  const void* v8;
  const float* q_scales;
  const float* k_scales;
  const float* v_scales;
  void* o;
  float* lse;
  int bh, n, d;
  float scale;
  int causal;
  int out_dtype;
  unsigned long long* err;
  unsigned long long* counter;
  cudaStream_t stream;
  int group = 1;
};
bool fwd_fp8_supported(int d);
cudaError_t launch_fwd_fp8(const Fp8FwdArgs& a);  // fwd_tc.cu: the 16-bit forward with 8-bit operands

// One CTA waits (bounded by timeout_ms) on an mbarrier phase nothing completes, or that it
// completes itself when arrive != 0.
cudaError_t launch_bounded_wait_selftest(unsigned long long* err, int timeout_ms, int arrive, cudaStream_t stream);

// One device index check, as debug builds make them: index outside [0, limit) is recorded.
cudaError_t launch_debug_check_selftest(unsigned long long* err, int index, int limit, cudaStream_t stream);

// Block b of `blocks` (one per SM when blocks <= the SM count) writes {SM id, SM cycle counter,
// global timer in ns} to out[3 b], out[3 b + 1], out[3 b + 2].
cudaError_t launch_sm_clock_sample(unsigned long long* out, int blocks, cudaStream_t stream);

// Records the calling thread's last error message (read by fa_last_error_message) and
// returns `status`.
int set_last_error(int status, const char* fmt, ...);

bool fwd_tc_supported(int dtype, int d);
bool bwd_tc_supported(int dtype, int d);
bool bwd_masked_fits(int group, int n, int d);  // masked backward's step list fits (tensor-core path)
bool fwd_masked_fits(int n, int d);             // masked forward's key-tile list fits

cudaError_t launch_fwd_tc(const FwdArgs& a);
cudaError_t launch_fwd_simt(const FwdArgs& a);
cudaError_t launch_bwd_pre(const BwdArgs& a);
cudaError_t launch_bwd_tc(const BwdArgs& a);
cudaError_t launch_bwd_simt(const BwdArgs& a);
cudaError_t launch_dq_convert(const BwdArgs& a);

}  // namespace fa
