// C ABI (include/fa.h): argument validation, workspace carving, kernel selection.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <mutex>

#include "fa.h"
#include "kernels.h"
#include "ptx.cuh"

namespace fa {
namespace {

// Device error word written by kernels (see ptx.cuh) and the tile counter.
__device__ unsigned long long g_err_word;
__device__ unsigned long long g_tile_counter;

thread_local char t_msg[512] = "";

fa_status fail(fa_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(t_msg, sizeof(t_msg), fmt, ap);
  va_end(ap);
  return s;
}

struct DeviceSyms {
  unsigned long long* err = nullptr;
  unsigned long long* counter = nullptr;
  unsigned long long ctx = 0;  // id of the context the addresses belong to
};

constexpr int kMaxDevices = 64;
DeviceSyms g_syms[kMaxDevices];
std::mutex g_syms_mu;

// Device addresses of the file-scope device symbols for the current device, looked up again
// whenever the current context is not the one they were taken in (a device reset destroys the
// primary context, and the next one may place the library's module elsewhere).
fa_status device_syms(DeviceSyms* out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(FA_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return fail(FA_ERR_UNSUPPORTED, "device index %d out of range", dev);
  std::lock_guard<std::mutex> lk(g_syms_mu);
  DeviceSyms& s = g_syms[dev];
  const unsigned long long ctx = current_context_id();
  if (!s.err || ctx == 0 || ctx != s.ctx) {
    void* p = nullptr;
    if ((e = cudaGetSymbolAddress(&p, g_err_word)) != cudaSuccess)
      return fail(FA_ERR_CUDA, "cudaGetSymbolAddress(error word): %s", cudaGetErrorString(e));
    void* c = nullptr;
    if ((e = cudaGetSymbolAddress(&c, g_tile_counter)) != cudaSuccess)
      return fail(FA_ERR_CUDA, "cudaGetSymbolAddress(tile counter): %s", cudaGetErrorString(e));
    s.counter = static_cast<unsigned long long*>(c);
    s.err = static_cast<unsigned long long*>(p);
    s.ctx = current_context_id();  // the lookup made the device's context current if none was
  }
  *out = s;
  return FA_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Shared shape/pointer checks. Returns FA_OK and sets *empty when there is nothing to do.
fa_status check_common(int B, int H, int N, int d, fa_dtype dt, bool* empty) {
  *empty = false;
  if (dt != FA_BF16 && dt != FA_FP16 && dt != FA_FP32) return fail(FA_ERR_UNSUPPORTED, "unknown dtype %d", (int)dt);
  if (B < 0 || H < 0 || N < 0) return fail(FA_ERR_INVALID_ARG, "negative size B=%d H=%d N=%d", B, H, N);
  if (d < 1 || d > 256) return fail(FA_ERR_UNSUPPORTED, "head dimension d=%d outside [1, 256]", d);
  const int64_t bh = (int64_t)B * H;
  if (bh > INT32_MAX) return fail(FA_ERR_INVALID_ARG, "B*H=%lld too large", (long long)bh);
  if ((int64_t)N > (int64_t)INT32_MAX - 128) return fail(FA_ERR_INVALID_ARG, "N=%d too large", N);
  const int64_t npad = padded_rows(N);
  if (bh > 0 && npad > 0 && (double)bh * (double)npad * (double)(d + 2) * 4.0 > 9.0e18)
    return fail(FA_ERR_INVALID_ARG, "problem too large");
  if (bh == 0 || N == 0) *empty = true;
  return FA_OK;
}

fa_status check_ptrs(std::initializer_list<const void*> ptrs, const char* what) {
  int i = 0;
  for (const void* p : ptrs) {
    if (!p) return fail(FA_ERR_INVALID_ARG, "%s: pointer %d is null", what, i);
    if (!aligned16(p)) return fail(FA_ERR_INVALID_ARG, "%s: pointer %d is not 16-byte aligned", what, i);
    ++i;
  }
  return FA_OK;
}

fa_status check_scale(float scale) {
  if (!std::isfinite(scale) || !(scale > 0.f)) return fail(FA_ERR_INVALID_ARG, "scale must be finite and > 0");
  return FA_OK;
}

fa_status launched(cudaError_t e, const char* what) {
  if (e != cudaSuccess) return fail(FA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
  t_msg[0] = 0;
  return FA_OK;
}

// A 16-bit call that had no tensor-core kernel and ran on the CUDA-core kernels: it succeeded,
// and the calling thread's message says which path ran (nothing changes backend silently).
fa_status note_cuda_core_path(fa_status st, const char* pass, fa_dtype dtype, int d) {
  if (st == FA_OK && dtype != FA_FP32)
    snprintf(t_msg, sizeof(t_msg),
             "notice: the %s %s pass at d=%d ran on the CUDA-core kernels (fp32 arithmetic): no tensor-core "
             "kernel for this head dimension",
             dtype == FA_BF16 ? "bf16" : "fp16", pass, d);
  return st;
}

// after the per-row vectors and the dQ accumulator: the backward's work-item queue counters
constexpr size_t kSchedBytes = 256;

size_t workspace_bytes_for(int B, int H, int N, int d) {
  const size_t bh = (size_t)B * H, npad = (size_t)padded_rows(N);
  return bh * npad * 4 * (2 + (size_t)d) + kSchedBytes;
}

fa_status carve(BwdArgs* a, void* ws, size_t ws_bytes, int B, int H, int N, int d) {
  const size_t need = workspace_bytes_for(B, H, N, d);
  if (ws_bytes < need) return fail(FA_ERR_INVALID_ARG, "workspace of %zu bytes < %zu required", ws_bytes, need);
  const size_t rows = (size_t)B * H * padded_rows(N);
  float* base = static_cast<float*>(ws);
  a->delta = base;
  a->lse2 = base + rows;
  a->dq_acc = base + 2 * rows;
  a->sched = reinterpret_cast<unsigned*>(base + rows * (2 + (size_t)d));
  return FA_OK;
}

}  // namespace

unsigned long long current_context_id() {
  static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
  static PFN_cuCtxGetId_v12000 get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
  });
  if (!get_current || !get_id) return 0;
  CUcontext c = nullptr;
  if (get_current(&c) != CUDA_SUCCESS || !c) return 0;
  unsigned long long id = 0;
  return get_id(c, &id) == CUDA_SUCCESS ? id : 0;
}

int device_sm_count() {
  static int cached[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return kSmCount;
  if (cached[dev] == 0) {
    int v = 0;
    cached[dev] = (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && v > 0) ? v : kSmCount;
  }
  return cached[dev];
}

int set_last_error(int status, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(t_msg, sizeof(t_msg), fmt, ap);
  va_end(ap);
  return status;
}

}  // namespace fa

using namespace fa;

namespace {

// Query heads H share key/value heads Hkv (H a multiple of Hkv); Hkv == H is plain attention.
fa_status check_heads(int H, int Hkv) {
  if (Hkv < 1 || H % Hkv != 0)
    return fail(FA_ERR_INVALID_ARG, "H=%d query heads must be a positive multiple of Hkv=%d key/value heads", H, Hkv);
  return FA_OK;
}

// Masks beyond causal: a window (keys with |i - j| >= window hidden; 0 = none) and a block
// mask of bytes [mask_heads][nb][nb] over 128 x 128 score blocks (NULL = none).
struct MaskSpec {
  int window = 0;
  const uint8_t* block_mask = nullptr;
  int mask_heads = 0;
  bool any() const { return window > 0 || block_mask != nullptr; }
};

fa_status check_mask(const MaskSpec& m, int H, int Hkv, int N, int d, fa_dtype dtype, bool backward) {
  if (m.window < 0) return fail(FA_ERR_INVALID_ARG, "window must be >= 0 (0: none), got %d", m.window);
  if (m.block_mask) {
    if (m.mask_heads != 1 && m.mask_heads != H)
      return fail(FA_ERR_INVALID_ARG, "mask_heads must be 1 or H=%d, got %d", H, m.mask_heads);
  } else if (m.mask_heads != 0) {
    return fail(FA_ERR_INVALID_ARG, "mask_heads=%d without a block mask (must be 0)", m.mask_heads);
  }
  if (!m.any()) return FA_OK;
  const bool tc = backward ? bwd_tc_supported((int)dtype, d) : fwd_tc_supported((int)dtype, d);
  if (!tc)
    return fail(FA_ERR_UNSUPPORTED, "block and window masks run on the tensor-core kernels (bf16/fp16, d in %s)",
                backward ? "{64, 128}" : "{64, 128, 256}");
  const bool fits = backward ? bwd_masked_fits(H / Hkv, N, d) : fwd_masked_fits(N, d);
  if (!fits) return fail(FA_ERR_UNSUPPORTED, "masked problem too long for the kernels' tile lists (N=%d)", N);
  return FA_OK;
}

fa_status fwd_impl(const void* Q, const void* K, const void* V, void* O, float* L, int B, int H, int Hkv, int N,
                   int d, float scale, int causal, fa_dtype dtype, void* stream, const char* name,
                   const MaskSpec& mask = MaskSpec()) {
  bool empty;
  fa_status st = check_common(B, H, N, d, dtype, &empty);
  if (st != FA_OK || empty) return st;
  if ((st = check_heads(H, Hkv)) != FA_OK) return st;
  if ((st = check_ptrs({Q, K, V, O, L}, name)) != FA_OK) return st;
  if ((st = check_scale(scale)) != FA_OK) return st;
  if ((st = check_mask(mask, H, Hkv, N, d, dtype, false)) != FA_OK) return st;
  DeviceSyms syms;
  if ((st = device_syms(&syms)) != FA_OK) return st;
  FwdArgs a{Q, K, V, O, L, B * H, N, d, scale, causal ? 1 : 0, (int)dtype, syms.err, syms.counter,
            static_cast<cudaStream_t>(stream)};
  a.group = H / Hkv;
  a.window = mask.window;
  a.block_mask = mask.block_mask;
  a.mask_heads = mask.mask_heads;
  a.heads = H;
  if (fwd_tc_supported(a.dtype, d)) return launched(launch_fwd_tc(a), "forward (tensor-core kernel)");
  return note_cuda_core_path(launched(launch_fwd_simt(a), "forward (CUDA-core kernel)"), "forward", dtype, d);
}

fa_status bwd_main_impl(const void* Q, const void* K, const void* V, const void* dO, void* dK, void* dV,
                        void* workspace, size_t workspace_bytes, int B, int H, int Hkv, int N, int d, float scale,
                        int causal, fa_dtype dtype, void* stream, const char* name, const MaskSpec& mask = MaskSpec()) {
  bool empty;
  fa_status st = check_common(B, H, N, d, dtype, &empty);
  if (st != FA_OK || empty) return st;
  if ((st = check_heads(H, Hkv)) != FA_OK) return st;
  if ((st = check_ptrs({Q, K, V, dO, dK, dV, workspace}, name)) != FA_OK) return st;
  if ((st = check_scale(scale)) != FA_OK) return st;
  if ((st = check_mask(mask, H, Hkv, N, d, dtype, true)) != FA_OK) return st;
  BwdArgs a{};
  if ((st = carve(&a, workspace, workspace_bytes, B, H, N, d)) != FA_OK) return st;
  DeviceSyms syms;
  if ((st = device_syms(&syms)) != FA_OK) return st;
  a.q = Q;
  a.k = K;
  a.v = V;
  a.dout = dO;
  a.dk = dK;
  a.dv = dV;
  a.bh = B * H;
  a.n = N;
  a.d = d;
  a.scale = scale;
  a.causal = causal ? 1 : 0;
  a.dtype = (int)dtype;
  a.err = syms.err;
  a.counter = syms.counter;
  a.stream = static_cast<cudaStream_t>(stream);
  a.group = H / Hkv;
  a.window = mask.window;
  a.block_mask = mask.block_mask;
  a.mask_heads = mask.mask_heads;
  a.heads = H;
  if (bwd_tc_supported(a.dtype, d)) return launched(launch_bwd_tc(a), "backward (tensor-core kernel)");
  return note_cuda_core_path(launched(launch_bwd_simt(a), "backward (CUDA-core kernels)"), "backward", dtype, d);
}

}  // namespace

extern "C" {

fa_status fa_fwd(const void* Q, const void* K, const void* V, void* O, float* L, int B, int H, int N, int d,
                 float scale, int causal, fa_dtype dtype, void* stream) {
  return fwd_impl(Q, K, V, O, L, B, H, H, N, d, scale, causal, dtype, stream, "fa_fwd");
}

fa_status fa_fwd_gqa(const void* Q, const void* K, const void* V, void* O, float* L, int B, int H, int Hkv, int N,
                     int d, float scale, int causal, fa_dtype dtype, void* stream) {
  return fwd_impl(Q, K, V, O, L, B, H, Hkv, N, d, scale, causal, dtype, stream, "fa_fwd_gqa");
}

size_t fa_bwd_workspace_size(int B, int H, int N, int d) {
  bool empty;
  if (check_common(B, H, N, d, FA_FP32, &empty) != FA_OK) return 0;
  return workspace_bytes_for(B, H, N, d);
}

fa_status fa_bwd_preprocess(const void* O, const void* dO, const float* L, void* workspace, size_t workspace_bytes,
                            int B, int H, int N, int d, fa_dtype dtype, void* stream) {
  bool empty;
  fa_status st = check_common(B, H, N, d, dtype, &empty);
  if (st != FA_OK || empty) return st;
  if ((st = check_ptrs({O, dO, L, workspace}, "fa_bwd_preprocess")) != FA_OK) return st;
  BwdArgs a{};
  if ((st = carve(&a, workspace, workspace_bytes, B, H, N, d)) != FA_OK) return st;
  a.o = O;
  a.dout = dO;
  a.lse = L;
  a.bh = B * H;
  a.n = N;
  a.d = d;
  a.dtype = (int)dtype;
  a.stream = static_cast<cudaStream_t>(stream);
  return launched(launch_bwd_pre(a), "fa_bwd_preprocess");
}

fa_status fa_bwd_main(const void* Q, const void* K, const void* V, const void* dO, void* dK, void* dV,
                      void* workspace, size_t workspace_bytes, int B, int H, int N, int d, float scale, int causal,
                      fa_dtype dtype, void* stream) {
  return bwd_main_impl(Q, K, V, dO, dK, dV, workspace, workspace_bytes, B, H, H, N, d, scale, causal, dtype, stream,
                       "fa_bwd_main");
}

fa_status fa_bwd_dq_convert(const void* workspace, size_t workspace_bytes, void* dQ, int B, int H, int N, int d,
                            float scale, fa_dtype dtype, void* stream) {
  bool empty;
  fa_status st = check_common(B, H, N, d, dtype, &empty);
  if (st != FA_OK || empty) return st;
  if ((st = check_ptrs({workspace, dQ}, "fa_bwd_dq_convert")) != FA_OK) return st;
  if ((st = check_scale(scale)) != FA_OK) return st;
  BwdArgs a{};
  if ((st = carve(&a, const_cast<void*>(workspace), workspace_bytes, B, H, N, d)) != FA_OK) return st;
  a.dq = dQ;
  a.bh = B * H;
  a.n = N;
  a.d = d;
  a.scale = scale;
  a.dtype = (int)dtype;
  a.stream = static_cast<cudaStream_t>(stream);
  return launched(launch_dq_convert(a), "fa_bwd_dq_convert");
}

fa_status fa_bwd_gqa(const void* Q, const void* K, const void* V, const void* O, const void* dO, const float* L,
                     void* dQ, void* dK, void* dV, void* workspace, size_t workspace_bytes, int B, int H, int Hkv,
                     int N, int d, float scale, int causal, fa_dtype dtype, void* stream) {
  bool empty;
  fa_status st = check_common(B, H, N, d, dtype, &empty);
  if (st != FA_OK || empty) return st;
  if ((st = check_heads(H, Hkv)) != FA_OK) return st;
  if ((st = check_ptrs({Q, K, V, O, dO, L, dQ, dK, dV, workspace}, "fa_bwd")) != FA_OK) return st;
  if ((st = check_scale(scale)) != FA_OK) return st;
  if ((st = fa_bwd_preprocess(O, dO, L, workspace, workspace_bytes, B, H, N, d, dtype, stream)) != FA_OK) return st;
  if ((st = bwd_main_impl(Q, K, V, dO, dK, dV, workspace, workspace_bytes, B, H, Hkv, N, d, scale, causal, dtype,
                          stream, "fa_bwd")) != FA_OK)
    return st;
  st = fa_bwd_dq_convert(workspace, workspace_bytes, dQ, B, H, N, d, scale, dtype, stream);
  return bwd_tc_supported((int)dtype, d) ? st : note_cuda_core_path(st, "backward", dtype, d);
}

fa_status fa_fwd_masked(const void* Q, const void* K, const void* V, void* O, float* L, int B, int H, int Hkv, int N,
                        int d, float scale, int causal, int window, const uint8_t* block_mask, int mask_heads,
                        fa_dtype dtype, void* stream) {
  MaskSpec m;
  m.window = window;
  m.block_mask = block_mask;
  m.mask_heads = mask_heads;
  return fwd_impl(Q, K, V, O, L, B, H, Hkv, N, d, scale, causal, dtype, stream, "fa_fwd_masked", m);
}

fa_status fa_bwd_masked(const void* Q, const void* K, const void* V, const void* O, const void* dO, const float* L,
                        void* dQ, void* dK, void* dV, void* workspace, size_t workspace_bytes, int B, int H, int Hkv,
                        int N, int d, float scale, int causal, int window, const uint8_t* block_mask, int mask_heads,
                        fa_dtype dtype, void* stream) {
  MaskSpec m;
  m.window = window;
  m.block_mask = block_mask;
  m.mask_heads = mask_heads;
  bool empty;
  fa_status st = check_common(B, H, N, d, dtype, &empty);
  if (st != FA_OK || empty) return st;
  if ((st = check_heads(H, Hkv)) != FA_OK) return st;
  if ((st = check_ptrs({Q, K, V, O, dO, L, dQ, dK, dV, workspace}, "fa_bwd_masked")) != FA_OK) return st;
  if ((st = check_scale(scale)) != FA_OK) return st;
  if ((st = check_mask(m, H, Hkv, N, d, dtype, true)) != FA_OK) return st;
  if ((st = fa_bwd_preprocess(O, dO, L, workspace, workspace_bytes, B, H, N, d, dtype, stream)) != FA_OK) return st;
  if ((st = bwd_main_impl(Q, K, V, dO, dK, dV, workspace, workspace_bytes, B, H, Hkv, N, d, scale, causal, dtype,
                          stream, "fa_bwd_masked", m)) != FA_OK)
    return st;
  return fa_bwd_dq_convert(workspace, workspace_bytes, dQ, B, H, N, d, scale, dtype, stream);
}

fa_status fa_bwd(const void* Q, const void* K, const void* V, const void* O, const void* dO, const float* L,
                 void* dQ, void* dK, void* dV, void* workspace, size_t workspace_bytes, int B, int H, int N, int d,
                 float scale, int causal, fa_dtype dtype, void* stream) {
  return fa_bwd_gqa(Q, K, V, O, dO, L, dQ, dK, dV, workspace, workspace_bytes, B, H, H, N, d, scale, causal, dtype,
                    stream);
}

// Effective number of cache splits: 0 or less picks automatically (for the kernel that runs);
// never more than Nk.
static int decode_splits(int B, int H, int Hkv, int Nq, int Nk, int d, int splits, bool tc) {
  int s = splits > 0 ? splits
                     : (tc ? decode_tc_auto_splits(B, H, Hkv, Nq, Nk, d) : decode_auto_splits(B, H, Hkv, Nq, Nk));
  if (s > Nk) s = Nk;
  if (s > 4096) s = 4096;
  return s < 1 ? 1 : s;
}

static fa_status check_decode(int B, int H, int Hkv, int Nq, int Nk, int d, fa_dtype dtype, bool* empty) {
  *empty = false;
  if (dtype != FA_BF16 && dtype != FA_FP16 && dtype != FA_FP32)
    return fail(FA_ERR_UNSUPPORTED, "unknown dtype %d", (int)dtype);
  if (B < 0 || H < 0 || Nq < 0 || Nk < 0) return fail(FA_ERR_INVALID_ARG, "negative size");
  if (d != 64 && d != 128 && d != 256) return fail(FA_ERR_UNSUPPORTED, "decode supports d in {64, 128, 256}, got %d", d);
  if ((int64_t)B * H * Nq == 0) {
    *empty = true;
    return FA_OK;
  }
  fa_status st = check_heads(H, Hkv);
  if (st != FA_OK) return st;
  if (Nk < 1) return fail(FA_ERR_INVALID_ARG, "decode needs at least one cached key (Nk=%d)", Nk);
  if ((double)B * Hkv * Nk * d > 4.0e15 || (double)B * H * Nq * d > 4.0e15)
    return fail(FA_ERR_INVALID_ARG, "problem too large");
  return FA_OK;
}

size_t fa_decode_workspace_size(int B, int H, int Hkv, int Nq, int Nk, int d, int splits) {
  bool empty;
  if (check_decode(B, H, Hkv, Nq, Nk, d, FA_BF16, &empty) != FA_OK || empty) return 0;
  // enough for either kernel (the size does not depend on the dtype)
  const int s = std::max(decode_splits(B, H, Hkv, Nq, Nk, d, splits, true), decode_splits(B, H, Hkv, Nq, Nk, d, splits, false));
  return decode_workspace_bytes(B, H, Nq, d, s);
}

fa_status fa_decode(const void* Q, const void* K, const void* V, void* O, float* L, int B, int H, int Hkv, int Nq,
                    int Nk, int d, float scale, int splits, fa_dtype dtype, void* workspace, size_t workspace_bytes,
                    void* stream) {
  bool empty;
  fa_status st = check_decode(B, H, Hkv, Nq, Nk, d, dtype, &empty);
  if (st != FA_OK || empty) return st;
  if ((st = check_ptrs({Q, K, V, O, L}, "fa_decode")) != FA_OK) return st;
  if ((st = check_scale(scale)) != FA_OK) return st;
  DecodeArgs a{};
  a.q = Q;
  a.k = K;
  a.v = V;
  a.o = O;
  a.lse = L;
  a.b = B;
  a.h = H;
  a.hkv = Hkv;
  a.nq = Nq;
  a.nk = Nk;
  a.d = d;
  a.scale = scale;
  const bool tc = decode_tc_supported((int)dtype, d, (int64_t)B * H * Nq);
  a.splits = decode_splits(B, H, Hkv, Nq, Nk, d, splits, tc);
  a.dtype = (int)dtype;
  a.stream = static_cast<cudaStream_t>(stream);
  DeviceSyms syms;
  if ((st = device_syms(&syms)) != FA_OK) return st;
  a.err = syms.err;
  a.counter = syms.counter;
  const size_t need = decode_workspace_bytes(B, H, Nq, d, a.splits);
  if (need > 0) {
    if (!workspace || !aligned16(workspace))
      return fail(FA_ERR_INVALID_ARG, "fa_decode: %d splits need a 16-byte-aligned workspace", a.splits);
    if (workspace_bytes < need)
      return fail(FA_ERR_INVALID_ARG, "fa_decode: workspace of %zu bytes < %zu required", workspace_bytes, need);
    a.ws = static_cast<float*>(workspace);
  }
  return launched(tc ? launch_decode_tc(a) : launch_decode(a), "fa_decode");
}

fa_status fa_quantize_fp8(const void* X, void* X8, float* scales, int B, int H, int N, int d, fa_dtype dtype,
                          void* stream) {
  bool empty;
  fa_status st = check_common(B, H, N, d, dtype, &empty);
  if (st != FA_OK || empty) return st;
  if (d != 64 && d != 128 && d != 256)
    return fail(FA_ERR_UNSUPPORTED, "fa_quantize_fp8 supports d in {64, 128, 256}, got %d", d);
  if ((st = check_ptrs({X, X8, scales}, "fa_quantize_fp8")) != FA_OK) return st;
  DeviceSyms syms;
  if ((st = device_syms(&syms)) != FA_OK) return st;
  QuantArgs a{X, X8, scales, B * H, N, d, (int)dtype, static_cast<cudaStream_t>(stream)};
  a.err = syms.err;
  return launched(launch_quantize_fp8(a), "fa_quantize_fp8");
}

fa_status fa_fwd_fp8_gqa(const void* Q8, const void* K8, const void* V8, const float* q_scales,
                         const float* k_scales, const float* v_scales, void* O, float* L, int B, int H, int Hkv, int N,
                         int d, float scale, int causal, fa_dtype out_dtype, void* stream) {
  if (out_dtype != FA_BF16 && out_dtype != FA_FP16)
    return fail(FA_ERR_UNSUPPORTED, "fa_fwd_fp8 writes O as bf16 or fp16, not dtype %d", (int)out_dtype);
  bool empty;
  fa_status st = check_common(B, H, N, d, out_dtype, &empty);
  if (st != FA_OK || empty) return st;
  if ((st = check_heads(H, Hkv)) != FA_OK) return st;
  if (!fwd_fp8_supported(d)) return fail(FA_ERR_UNSUPPORTED, "fa_fwd_fp8 supports d in {64, 128, 256}, got %d", d);
  if ((st = check_ptrs({Q8, K8, V8, q_scales, k_scales, v_scales, O, L}, "fa_fwd_fp8")) != FA_OK) return st;
  if ((st = check_scale(scale)) != FA_OK) return st;
  DeviceSyms syms;
  if ((st = device_syms(&syms)) != FA_OK) return st;
  Fp8FwdArgs a{};
  a.q8 = Q8;
  a.k8 = K8;
  a.v8 = V8;
  a.q_scales = q_scales;
  a.k_scales = k_scales;
  a.v_scales = v_scales;
  a.o = O;
  a.lse = L;
  a.bh = B * H;
  a.n = N;
  a.d = d;
  a.scale = scale;
  a.causal = causal ? 1 : 0;
  a.out_dtype = (int)out_dtype;
  a.err = syms.err;
  a.counter = syms.counter;
  a.stream = static_cast<cudaStream_t>(stream);
  a.group = H / Hkv;
  return launched(launch_fwd_fp8(a), "fa_fwd_fp8");
}

fa_status fa_fwd_fp8(const void* Q8, const void* K8, const void* V8, const float* q_scales, const float* k_scales,
                     const float* v_scales, void* O, float* L, int B, int H, int N, int d, float scale, int causal,
                     fa_dtype out_dtype, void* stream) {
  return fa_fwd_fp8_gqa(Q8, K8, V8, q_scales, k_scales, v_scales, O, L, B, H, H, N, d, scale, causal, out_dtype,
                        stream);
}

fa_status fa_check_device_error(void* stream) {
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(FA_ERR_CUDA, "stream synchronize: %s", cudaGetErrorString(e));
  DeviceSyms syms;
  fa_status st = device_syms(&syms);
  if (st != FA_OK) return st;
  unsigned long long w = 0;
  if ((e = cudaMemcpy(&w, syms.err, sizeof(w), cudaMemcpyDeviceToHost)) != cudaSuccess)
    return fail(FA_ERR_CUDA, "reading the device error word: %s", cudaGetErrorString(e));
  if (w == 0) {
    t_msg[0] = 0;
    return FA_OK;
  }
  const unsigned long long zero = 0;
  cudaMemcpy(syms.err, &zero, sizeof(zero), cudaMemcpyHostToDevice);
  const unsigned code = (unsigned)(w >> 56), site = (unsigned)((w >> 40) & 0xFFFF);
  const unsigned long long block = w & 0xFFFFFFFFFFull;
  if (code == DERR_TIMEOUT)
    return fail(FA_ERR_TIMEOUT, "a bounded wait expired (site %u, block %llu)", site, block);
  if (code == DERR_BOUNDS)
    return fail(FA_ERR_DEVICE, "device index check failed (site %u, block %llu)", site, block);
  return fail(FA_ERR_DEVICE, "device check %u failed (site %u, block %llu)", code, site, block);
}

fa_status fa_selftest_bounded_wait(int timeout_ms, int arrive, void* stream) {
  if (timeout_ms < 1 || timeout_ms > 1000)
    return fail(FA_ERR_INVALID_ARG, "fa_selftest_bounded_wait: timeout_ms must be in [1, 1000], got %d", timeout_ms);
  DeviceSyms syms;
  fa_status st = device_syms(&syms);
  if (st != FA_OK) return st;
  return launched(launch_bounded_wait_selftest(syms.err, timeout_ms, arrive ? 1 : 0, static_cast<cudaStream_t>(stream)),
                  "fa_selftest_bounded_wait");
}

fa_status fa_selftest_debug_check(int index, int limit, void* stream) {
  if (!FA_DEBUG_CHECKS) return fail(FA_ERR_UNSUPPORTED, "fa_selftest_debug_check: library built without FA_DEBUG");
  DeviceSyms syms;
  fa_status st = device_syms(&syms);
  if (st != FA_OK) return st;
  return launched(launch_debug_check_selftest(syms.err, index, limit, static_cast<cudaStream_t>(stream)),
                  "fa_selftest_debug_check");
}

int fa_debug_build(void) { return FA_DEBUG_CHECKS; }

fa_status fa_sm_clock_sample(unsigned long long* out, int blocks, void* stream) {
  if (!out || !aligned16(out)) return fail(FA_ERR_INVALID_ARG, "fa_sm_clock_sample: null or misaligned output");
  if (blocks < 1 || blocks > device_sm_count())
    return fail(FA_ERR_INVALID_ARG, "fa_sm_clock_sample: blocks=%d outside [1, %d]", blocks, device_sm_count());
  return launched(launch_sm_clock_sample(out, blocks, static_cast<cudaStream_t>(stream)), "fa_sm_clock_sample");
}

fa_status fa_tile_counter(void* stream, unsigned long long* value, int reset) {
  if (!value) return fail(FA_ERR_INVALID_ARG, "fa_tile_counter: null output");
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(FA_ERR_CUDA, "stream synchronize: %s", cudaGetErrorString(e));
  DeviceSyms syms;
  fa_status st = device_syms(&syms);
  if (st != FA_OK) return st;
  if ((e = cudaMemcpy(value, syms.counter, sizeof(*value), cudaMemcpyDeviceToHost)) != cudaSuccess)
    return fail(FA_ERR_CUDA, "reading the tile counter: %s", cudaGetErrorString(e));
  if (reset) {
    const unsigned long long zero = 0;
    if ((e = cudaMemcpy(syms.counter, &zero, sizeof(zero), cudaMemcpyHostToDevice)) != cudaSuccess)
      return fail(FA_ERR_CUDA, "resetting the tile counter: %s", cudaGetErrorString(e));
  }
  return FA_OK;
}

int fa_uses_tensor_cores(int pass, fa_dtype dtype, int d) {
  return pass == 0 ? (int)fwd_tc_supported((int)dtype, d) : (int)bwd_tc_supported((int)dtype, d);
}

const char* fa_status_string(fa_status s) {
  switch (s) {
    case FA_OK: return "ok";
    case FA_ERR_INVALID_ARG: return "invalid argument";
    case FA_ERR_UNSUPPORTED: return "unsupported dtype or head dimension";
    case FA_ERR_CUDA: return "CUDA error";
    case FA_ERR_TIMEOUT: return "device wait timed out";
    case FA_ERR_DEVICE: return "device-side check failed";
  }
  return "unknown status";
}

const char* fa_last_error_message(void) { return t_msg; }

}  // extern "C"
