/*
 * fa.h — C ABI of the exact tiled attention library for NVIDIA GB300 (sm_103a).
 *
 * The operation is exact scaled-dot-product attention computed tile by tile with an
 * online softmax, so the N x N score matrix S and probability matrix P never reach
 * device memory:
 *
 *   forward   O = softmax(scale * Q K^T [+ causal mask]) V,   L_i = m_i + ln l_i
 *   backward  dQ, dK, dV of f = sum(O o dO), recomputing S and P block by block from
 *             Q, K and L, with D_i = sum_k dO_ik O_ik precomputed
 *
 * Sources (page title, section): "Lecture 8 · GPU Performance & FlashAttention"
 * (CS324 notes) §5.1 standard attention, §5.2 online softmax, §5.3 tiled forward and
 * causal block skipping, §5.4 recomputing backward and the D identity, §8.1 FA2 work
 * split; "FlashAttention and GPU memory" (world.lapla.si explainer) §07–§09.
 *
 * Conventions shared by every entry point
 *   Layout    Q, K, V, O, dO, dQ, dK, dV: contiguous row-major [B][H][N][d] of the
 *             element type `dtype` (one N x d matrix per head). L: fp32 [B][H][N],
 *             natural-log units. Keys and queries have the same length N.
 *   Causal    causal != 0 masks key j for query i when j > i (top-left aligned).
 *   Memory    All pointers are DEVICE pointers owned by the caller; the library keeps no
 *             per-call allocation and never allocates anything N x N. Every pointer
 *             must be 16-byte aligned. Buffers must not overlap, except that the
 *             library only reads Q, K, V, O, dO and L.
 *   Streams   `stream` is a cudaStream_t (NULL = legacy default stream). Calls are
 *             asynchronous: they validate, enqueue kernels on `stream` and return.
 *   Errors    Invalid arguments return an error and launch nothing. Device-side
 *             failures (a bounded wait that timed out) are recorded in a library error
 *             word and reported by fa_check_device_error. No C++ exception crosses
 *             this interface. fa_last_error_message() describes the last failure of
 *             the calling thread.
 *   Paths     bf16/fp16 with d in {64, 128, 256} run the tensor-core kernels (TMA,
 *             tcgen05 MMAs accumulating in tensor memory), forward and backward; fp32, and
 *             any other d in [1, 256], run CUDA-core kernels that compute in fp32. The
 *             choice is never silent: fa_uses_tensor_cores() tells it in advance, and a
 *             bf16/fp16 call that runs on the CUDA-core kernels (another d) returns FA_OK
 *             with a notice in fa_last_error_message() naming the path that ran.
 */
#ifndef FA_H_
#define FA_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define FA_API __attribute__((visibility("default")))
#else
#define FA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { FA_BF16 = 0, FA_FP16 = 1, FA_FP32 = 2 } fa_dtype;

typedef enum {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = 1, /* null/misaligned pointer, bad size, scale not finite and > 0 */
  FA_ERR_UNSUPPORTED = 2, /* dtype or head dimension outside what any kernel handles */
  FA_ERR_CUDA = 3,        /* a CUDA runtime call or kernel launch failed */
  FA_ERR_TIMEOUT = 4,     /* a kernel's bounded wait expired (reported by fa_check_device_error) */
  FA_ERR_DEVICE = 5       /* another device-side check failed (reported by fa_check_device_error) */
} fa_status;

/*
 * Forward pass ("Lecture 8" §5.3; FA2 order §8.1).
 *   Q, K, V   in:  [B][H][N][d] dtype
 *   O         out: [B][H][N][d] dtype, softmax(scale Q K^T [+mask]) V
 *   L         out: [B][H][N] fp32, row log-sum-exp of the (masked) scaled scores
 *   B, H, N   >= 0 (an empty problem returns FA_OK without launching); d in [1, 256]
 *   scale     the factor tau on Q K^T, finite and > 0 (usually 1/sqrt(d))
 * Launches one kernel.
 */
FA_API fa_status fa_fwd(const void* Q, const void* K, const void* V, void* O, float* L, int B, int H, int N, int d,
                 float scale, int causal, fa_dtype dtype, void* stream);

/*
 * Forward pass with grouped-query / multi-query attention ("Lecture 8" §8.2): H query heads
 * share Hkv key/value heads, query head h of a batch row reading key/value head
 * h / (H / Hkv). K and V are [B][Hkv][N][d]; Q, O are [B][H][N][d]; L is [B][H][N].
 * H must be a positive multiple of Hkv (Hkv == 1: multi-query; Hkv == H: fa_fwd).
 */
FA_API fa_status fa_fwd_gqa(const void* Q, const void* K, const void* V, void* O, float* L, int B, int H, int Hkv,
                            int N, int d, float scale, int causal, fa_dtype dtype, void* stream);

/*
 * Bytes of device workspace fa_bwd needs: per head, with Np = N rounded up to 128,
 * D [Np] fp32, L*log2(e) [Np] fp32 and an fp32 dQ accumulator [Np][d]; then 256 bytes for
 * the counters of the tensor-core backward's work-item queue.
 * Returns 0 for invalid sizes.
 */
FA_API size_t fa_bwd_workspace_size(int B, int H, int N, int d);

/*
 * Backward pass with recomputation ("Lecture 8" §5.4): the three stages below in order.
 *   Q, K, V, O, dO  in:  [B][H][N][d] dtype (O from fa_fwd)
 *   L               in:  [B][H][N] fp32 from fa_fwd
 *   dQ, dK, dV      out: [B][H][N][d] dtype
 *   workspace       scratch of at least fa_bwd_workspace_size(B, H, N, d) bytes, 16-byte
 *                   aligned, owned by the caller; its contents on entry do not matter.
 * Launches three kernels (preprocess, main, dQ conversion).
 */
FA_API fa_status fa_bwd(const void* Q, const void* K, const void* V, const void* O, const void* dO, const float* L,
                 void* dQ, void* dK, void* dV, void* workspace, size_t workspace_bytes, int B, int H, int N, int d,
                 float scale, int causal, fa_dtype dtype, void* stream);

/*
 * Backward pass with grouped-query / multi-query attention: as fa_bwd, with K, V, dK, dV of
 * Hkv heads ([B][Hkv][N][d]). dK and dV of a key/value head are the sums over the query heads
 * that read it (the gradient of a shared operand). The workspace is the one of
 * fa_bwd_workspace_size(B, H, N, d) (per query head). Launches three kernels.
 */
FA_API fa_status fa_bwd_gqa(const void* Q, const void* K, const void* V, const void* O, const void* dO,
                            const float* L, void* dQ, void* dK, void* dV, void* workspace, size_t workspace_bytes,
                            int B, int H, int Hkv, int N, int d, float scale, int causal, fa_dtype dtype,
                            void* stream);

/*
 * Stage 1 of fa_bwd: D_i = sum_k dO_ik O_ik (the N x d identity that replaces the N x N
 * row sum of P o dP, "Lecture 8" §5.4), L_i log2(e) for the exp2-domain recomputation,
 * a zeroed dQ accumulator and zeroed work-queue counters, all into `workspace`.
 */
FA_API fa_status fa_bwd_preprocess(const void* O, const void* dO, const float* L, void* workspace, size_t workspace_bytes,
                            int B, int H, int N, int d, fa_dtype dtype, void* stream);

/*
 * Stage 2 of fa_bwd: recompute S and P block by block and produce dK, dV (written) and
 * the unscaled dQ sum (accumulated in `workspace`). Needs stage 1 on the same workspace.
 * The tensor-core kernel's CTAs draw work items from the queue counters, which stage 1 set
 * to zero and which this stage leaves at zero when it completes; two calls must not run at
 * the same time on one workspace.
 */
FA_API fa_status fa_bwd_main(const void* Q, const void* K, const void* V, const void* dO, void* dK, void* dV,
                      void* workspace, size_t workspace_bytes, int B, int H, int N, int d, float scale, int causal,
                      fa_dtype dtype, void* stream);

/* Stage 3 of fa_bwd: dQ = scale * (dQ accumulator), converted to dtype. */
FA_API fa_status fa_bwd_dq_convert(const void* workspace, size_t workspace_bytes, void* dQ, int B, int H, int N, int d,
                            float scale, fa_dtype dtype, void* stream);

/*
 * Backward pass for callers that cannot allocate device memory: the same computation and
 * arguments as fa_bwd, without `workspace`. (The pages have no counterpart of this entry
 * point; it exists for the library's callers.)
 *
 * Some callers cannot provide a workspace: code inside a host application that owns every
 * device allocation (a plugin or runtime with its own memory pool), or a latency-bound
 * loop that cannot afford cudaMalloc's implicit device synchronisation. This entry point
 * takes its scratch from a static device array of FA_BWD_NOALLOC_SCRATCH_BYTES that the
 * library holds on every GPU where it is loaded, until the process exits. It calls no
 * cudaMalloc, cudaFree or other allocating routine.
 *
 *   Limit     fa_bwd_workspace_size(B, H, N, d) must not exceed FA_BWD_NOALLOC_SCRATCH_BYTES;
 *             larger problems return FA_ERR_INVALID_ARG and launch nothing.
 *   Set-up    The first call on a device looks up the array's device address
 *             (cudaGetSymbolAddress) with that device current; make that first call
 *             before any stream capture. (If the device's context is destroyed and
 *             recreated, e.g. by cudaDeviceReset, the next call looks it up again.)
 *   Sharing   Every call uses the same array and leaves its contents behind; each call
 *             re-initialises what it reads. Calls whose kernels overlap on the GPU
 *             (different streams or host threads) race on the array: serialise them.
 */
#define FA_BWD_NOALLOC_SCRATCH_BYTES (64ull << 20)
FA_API fa_status fa_bwd_noalloc(const void* Q, const void* K, const void* V, const void* O, const void* dO,
                                const float* L, void* dQ, void* dK, void* dV, int B, int H, int N, int d, float scale,
                                int causal, fa_dtype dtype, void* stream);

/*
 * Forward and backward with every tensor in HOST memory (Q, K, V, dO in; O, L, dQ, dK, dV
 * out; the layouts of fa_fwd_gqa / fa_bwd_gqa): the computation of fa_fwd_gqa followed by
 * fa_bwd_gqa, with the copies between host and device done here. Attention heads are
 * independent ("Lecture 8" §5.1: one N x d problem per head), so the batch is cut into chunks
 * of key/value heads (each with its H / Hkv query heads) that are copied in, computed and
 * copied out on three internal streams: the copies of one chunk overlap the computation of
 * its neighbours. (The pages have no counterpart of this entry point; it exists for callers
 * whose data is in host memory.)
 *   chunk      key/value heads per chunk (counted over B x Hkv); 0 chooses about eight chunks
 *   workspace  device scratch of fa_fwd_bwd_host_workspace_size(...) bytes for the same
 *              arguments, 256-byte aligned, owned by the caller (two slots of chunk buffers)
 *   stream     the call is ordered after earlier work on `stream`, and work enqueued on
 *              `stream` afterwards runs after its last copy out; the host does not wait.
 *              Host buffers must stay valid (and, for the copies to overlap, page-locked)
 *              until then.
 * Calls from several host threads on one device are serialised on the internal streams.
 */
FA_API size_t fa_fwd_bwd_host_workspace_size(int B, int H, int Hkv, int N, int d, fa_dtype dtype, int chunk);
FA_API fa_status fa_fwd_bwd_host(const void* Q, const void* K, const void* V, const void* dO, void* O, float* L,
                                 void* dQ, void* dK, void* dV, void* workspace, size_t workspace_bytes, int B, int H,
                                 int Hkv, int N, int d, float scale, int causal, fa_dtype dtype, int chunk,
                                 void* stream);

/*
 * Decode attention over a key/value cache with the cache split across thread blocks
 * ("Lecture 8" §8.2: the cache is cut into pieces processed in parallel and the partial
 * results are combined with the online-softmax merge of Exercise 3).
 *   Q        in:  [B][H][Nq][d] dtype, the new query rows
 *   K, V     in:  [B][Hkv][Nk][d] dtype, the cache (H a multiple of Hkv; query head h reads
 *                 key/value head h / (H / Hkv))
 *   O, L     out: [B][H][Nq][d] dtype and [B][H][Nq] fp32; every query row attends to all Nk
 *                 cached keys (no mask)
 *   d        64, 128 or 256; Nk >= 1
 *   splits   number of cache pieces; <= 0 chooses automatically; capped at Nk
 *   workspace  fa_decode_workspace_size(...) bytes for the same arguments (0 when there is a
 *            single piece: then workspace may be NULL)
 * Launches one kernel, plus one merge kernel when there is more than one piece. bf16/fp16 run
 * on the tensor cores (the rows sharing a key/value head form one 128-row tile), fp32 on CUDA
 * cores; either way each cached key and value is read once and the call is bound by HBM
 * bandwidth. The size fa_decode_workspace_size returns covers every dtype.
 */
FA_API size_t fa_decode_workspace_size(int B, int H, int Hkv, int Nq, int Nk, int d, int splits);
FA_API fa_status fa_decode(const void* Q, const void* K, const void* V, void* O, float* L, int B, int H, int Hkv,
                           int Nq, int Nk, int d, float scale, int splits, fa_dtype dtype, void* workspace,
                           size_t workspace_bytes, void* stream);

/*
 * Attention with a block-sparse mask and/or a sliding window ("Lecture 8" §5.7: block-sparse
 * FlashAttention computes only the non-zero B_r x B_c blocks of S, and reads, writes and FLOPs
 * fall in proportion, Proposition 4; the sliding window is the local approximation).
 * Key j is visible to query i when all of these hold:
 *   block_mask  NULL, or byte [i / 128][j / 128] of the head's [nb][nb] mask is non-zero
 *               (nb = ceil(N / 128); device memory, mask_heads masks of nb * nb bytes:
 *               mask_heads = 1 shares one mask, mask_heads = H gives one per query head;
 *               mask_heads must be 0 when block_mask is NULL)
 *   causal      j <= i (when causal != 0)
 *   window      |i - j| < window (when window > 0; with causal: the last `window` positions)
 * A row that sees no key gets O = 0 and L = -inf and contributes nothing to the gradients.
 * Blocks with no visible score are never loaded or multiplied. Other arguments, layouts and
 * errors as fa_fwd_gqa / fa_bwd_gqa. Runs on the tensor-core kernels only: bf16/fp16 with
 * d in {64, 128, 256} (forward) or {64, 128} (backward); other dtypes or head dims return
 * FA_ERR_UNSUPPORTED, as does a sequence whose tile list does not fit in shared memory
 * (forward: N up to about 1.5M; backward: H/Hkv <= 16 and N <= 524,288, less when the
 * query heads per key/value head times N/128 passes about 4,000 for d = 128).
 */
FA_API fa_status fa_fwd_masked(const void* Q, const void* K, const void* V, void* O, float* L, int B, int H, int Hkv,
                               int N, int d, float scale, int causal, int window, const uint8_t* block_mask,
                               int mask_heads, fa_dtype dtype, void* stream);
FA_API fa_status fa_bwd_masked(const void* Q, const void* K, const void* V, const void* O, const void* dO,
                               const float* L, void* dQ, void* dK, void* dV, void* workspace, size_t workspace_bytes,
                               int B, int H, int Hkv, int N, int d, float scale, int causal, int window,
                               const uint8_t* block_mask, int mask_heads, fa_dtype dtype, void* stream);

/*
 * FP8 (E4M3) block quantisation ("Lecture 8" §8.1, "FlashAttention and GPU memory" §11: the
 * third generation runs attention in 8-bit floating point with one scale per block).
 *   X        in:  [B][H][N][d] dtype (bf16, fp16 or fp32)
 *   X8       out: [B][H][N][d] bytes, E4M3 codes (1 sign, 4 exponent bits with bias 7,
 *                 3 mantissa bits; largest finite value 448)
 *   scales   out: [B][H][ceil(N / 128)] fp32; block b of a head is rows [128 b, 128 b + 128)
 *   d        64, 128 or 256
 * For each block, scale = amax / 448 (1 when the block is all zero) and
 * code = E4M3(x / scale), rounded to nearest even and saturated at +-448; both divisions are
 * fp32 divisions rounded to nearest. One kernel launch: for 16-bit inputs a persistent grid
 * (three thread blocks per SM) streams the blocks; for fp32 inputs one thread block takes one
 * block.
 */
FA_API fa_status fa_quantize_fp8(const void* X, void* X8, float* scales, int B, int H, int N, int d, fa_dtype dtype,
                                 void* stream);

/*
 * Forward attention on FP8 inputs with block scales (tensor cores, kind::f8f6f4).
 *   Q8, K8, V8           in:  [B][H][N][d] E4M3 codes, as written by fa_quantize_fp8
 *   q/k/v_scales         in:  [B][H][ceil(N / 128)] fp32 block scales
 *   O                    out: [B][H][N][d] out_dtype (FA_BF16 or FA_FP16)
 *   L                    out: [B][H][N] fp32, natural-log log-sum-exp of the scaled scores
 *   d                    64, 128 or 256 (other head dims return FA_ERR_UNSUPPORTED)
 * Computes attention of the dequantised tensors (code x block scale): S = scale Q K^T (causal
 * mask when causal != 0), O = softmax(S) V, L = m + ln l. The probabilities are rounded to
 * E4M3 before the P V product, after multiplying by the key block's V scale; the online
 * softmax's running maximum includes that factor, so a row's largest weighted probabilities
 * stay near 1 whatever the spread of the V scales. O carries E4M3's relative rounding of P (at
 * most 2^-4 per element above E4M3's subnormal range); L does not. Pointers 16-byte aligned; the same errors as fa_fwd.
 */
FA_API fa_status fa_fwd_fp8(const void* Q8, const void* K8, const void* V8, const float* q_scales,
                            const float* k_scales, const float* v_scales, void* O, float* L, int B, int H, int N,
                            int d, float scale, int causal, fa_dtype out_dtype, void* stream);

/*
 * fa_fwd_fp8 with grouped-query / multi-query attention: K8, V8 and their block scales hold
 * Hkv heads ([B][Hkv][N][d], [B][Hkv][ceil(N / 128)]); query head h reads key/value head
 * h / (H / Hkv). H must be a positive multiple of Hkv.
 */
FA_API fa_status fa_fwd_fp8_gqa(const void* Q8, const void* K8, const void* V8, const float* q_scales,
                                const float* k_scales, const float* v_scales, void* O, float* L, int B, int H,
                                int Hkv, int N, int d, float scale, int causal, fa_dtype out_dtype, void* stream);

/*
 * Synchronises `stream` and reports device-side failures of earlier calls on the
 * current device: FA_ERR_CUDA for a CUDA error, FA_ERR_TIMEOUT / FA_ERR_DEVICE for a
 * failure a kernel recorded. The recorded failure is cleared.
 */
FA_API fa_status fa_check_device_error(void* stream);

/*
 * Self-test of failure detection without a GPU fault: launches one thread block that waits on
 * an mbarrier phase, through the same bounded wait every kernel uses, with a limit of
 * timeout_ms (1..1000). With arrive == 0 nothing completes the phase: the wait gives up after
 * timeout_ms, records a timeout in the device error word and the kernel returns, so the next
 * fa_check_device_error returns FA_ERR_TIMEOUT and the context stays usable. With arrive != 0
 * the block completes the phase itself and nothing is recorded.
 */
FA_API fa_status fa_selftest_bounded_wait(int timeout_ms, int arrive, void* stream);

/*
 * Debug builds. The library built with FA_DEBUG (exact_tiled_attention_07_gb300/build.py,
 * debug=True: libfa_gb300_debug.so) checks work-item, tile and row indices inside the kernels;
 * a failed check records a device error (fa_check_device_error: FA_ERR_DEVICE, "device index
 * check failed"), stops the kernel's roles through their bounded waits and never traps.
 * fa_debug_build() is 1 in such a library, 0 otherwise. fa_selftest_debug_check launches one
 * such check of index against [0, limit) (a debug build records a failure when it is outside);
 * a release build returns FA_ERR_UNSUPPORTED.
 */
FA_API int fa_debug_build(void);
FA_API fa_status fa_selftest_debug_check(int index, int limit, void* stream);

/*
 * Diagnostic: number of (query tile, key tile) pairs the forward kernels processed on the
 * current device since the last reset (128 x 128 tiles on the tensor-core path, 32 x 32 on
 * the CUDA-core path); skipped causal tiles are not counted. Synchronises `stream`;
 * reset != 0 clears the counter afterwards.
 */
FA_API fa_status fa_tile_counter(void* stream, unsigned long long* value, int reset);

/*
 * Measurement helper (no counterpart on the pages): launches `blocks` thread blocks on `stream`
 * (1 <= blocks <= the device's SM count; each takes enough shared memory to have an SM to
 * itself) and block b writes three 64-bit words to the DEVICE array out[3 * blocks]:
 * out[3 b] = the id of the SM it ran on, out[3 b + 1] = that SM's cycle counter (%clock64),
 * out[3 b + 2] = the global timer in nanoseconds (%globaltimer). Two samples taken on a stream
 * before and after a stretch of work give, for each SM seen in both, its mean clock over that
 * stretch: (cycles difference) / (nanoseconds difference) GHz.
 */
FA_API fa_status fa_sm_clock_sample(unsigned long long* out, int blocks, void* stream);

/* Whether the given pass ("fwd" = 0, "bwd" = 1) runs on tensor cores for dtype and d. */
FA_API int fa_uses_tensor_cores(int pass, fa_dtype dtype, int d);

/* Static text for a status code. */
FA_API const char* fa_status_string(fa_status status);

/* Description of the last failure on the calling thread ("" if none), or, after a successful
 * 16-bit call that ran on the CUDA-core kernels, a notice saying so (starting "notice:"). */
FA_API const char* fa_last_error_message(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_H_ */
