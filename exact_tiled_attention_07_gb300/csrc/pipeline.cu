// fa_fwd_bwd_host: forward and backward over host buffers.
//
// A caller whose Q, K, V, dO live in host memory, and who wants O, L, dQ, dK, dV back there,
// would otherwise copy everything in, compute, and copy everything out, one after the other:
// for the causal LM shape (B=8, H=16, N=4096, d=128) the 1.08 GB of copies take three times
// as long as the computation.  Attention heads are independent, so the batch is cut into
// chunks of key/value heads (each with its group of query heads), and chunk c is copied in
// (stream `in`), computed (stream `comp`: fa_fwd_gqa, then fa_bwd_gqa) and copied out (stream
// `out`) while chunk c + 1 is copied in and chunk c - 1 copied out.  Two slots of device
// buffers, in the caller's workspace, alternate between chunks; events keep a slot's inputs
// until its computation has read them and its outputs until they have been copied out.
//
// The three streams and their events are created once per device and shared by every call;
// a mutex serialises callers, and each call waits for the previous one's work on them before
// reusing a slot.  The call is ordered after earlier work on the caller's stream and the
// caller's stream waits for its last copy out; the host does not wait.
#include <cuda_runtime.h>
#include <algorithm>
#include <cstdint>
#include <mutex>

#include "fa.h"
#include "kernels.h"

namespace fa {
namespace {

constexpr int kMaxDevices = 64;
constexpr size_t kAlign = 256;

size_t round_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

// Device buffers of one slot, for a chunk of `units` key/value heads of `g` query heads each.
struct Slot {
  size_t q, k, v, dout, o, lse, dq, dk, dv, ws, ws_bytes, total;
};

Slot slot_layout(int units, int g, int N, int d, int eb) {
  Slot s{};
  const size_t hq = (size_t)units * g, hk = (size_t)units;
  const size_t mq = hq * N * d * eb, mk = hk * N * d * eb;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off += round_up(bytes);
    return at;
  };
  s.q = take(mq);
  s.k = take(mk);
  s.v = take(mk);
  s.dout = take(mq);
  s.o = take(mq);
  s.lse = take(hq * N * 4);
  s.dq = take(mq);
  s.dk = take(mk);
  s.dv = take(mk);
  s.ws_bytes = fa_bwd_workspace_size(1, (int)hq, N, d);
  s.ws = take(s.ws_bytes);
  s.total = off;
  return s;
}

// key/value heads per chunk: `chunk` if positive (at most all of them), else about eight chunks
int chunk_units(int units, int chunk) { return chunk > 0 ? std::min(chunk, units) : std::max(1, (units + 7) / 8); }

struct Pipe {
  cudaStream_t in = nullptr, comp = nullptr, out = nullptr;
  cudaEvent_t start = nullptr, fin = nullptr, in_end = nullptr, comp_end = nullptr;
  cudaEvent_t in_ready[2] = {}, comp_done[2] = {}, out_done[2] = {};
  bool used = false;  // fin holds the end of a previous call
};
Pipe g_pipe[kMaxDevices];
std::mutex g_pipe_mu[kMaxDevices];

fa_status cuda_fail(cudaError_t e, const char* what) {
  return (fa_status)set_last_error(FA_ERR_CUDA, "fa_fwd_bwd_host: %s: %s", what, cudaGetErrorString(e));
}

// streams and events of this device, created on first use
fa_status pipe_init(Pipe& p) {
  if (p.in) return FA_OK;
  cudaError_t e = cudaSuccess;
  for (cudaStream_t* s : {&p.in, &p.comp, &p.out})
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(s, cudaStreamNonBlocking);
  for (cudaEvent_t* ev : {&p.start, &p.fin, &p.in_end, &p.comp_end, &p.in_ready[0], &p.in_ready[1], &p.comp_done[0],
                          &p.comp_done[1], &p.out_done[0], &p.out_done[1]})
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
  if (e != cudaSuccess) return cuda_fail(e, "creating streams and events");
  return FA_OK;
}

fa_status check_args(int B, int H, int Hkv, int N, int d, fa_dtype dtype, int chunk) {
  if (dtype != FA_BF16 && dtype != FA_FP16 && dtype != FA_FP32)
    return (fa_status)set_last_error(FA_ERR_UNSUPPORTED, "fa_fwd_bwd_host: unknown dtype %d", (int)dtype);
  if (B < 0 || H < 0 || N < 0 || chunk < 0)
    return (fa_status)set_last_error(FA_ERR_INVALID_ARG, "fa_fwd_bwd_host: negative size");
  if (Hkv < 1 || H % Hkv != 0)
    return (fa_status)set_last_error(FA_ERR_INVALID_ARG,
                                     "fa_fwd_bwd_host: H=%d must be a positive multiple of Hkv=%d", H, Hkv);
  if (d < 1 || d > 256)
    return (fa_status)set_last_error(FA_ERR_UNSUPPORTED, "fa_fwd_bwd_host: head dimension d=%d outside [1, 256]", d);
  if ((int64_t)B * H > INT32_MAX || (int64_t)N > (int64_t)INT32_MAX - 128)
    return (fa_status)set_last_error(FA_ERR_INVALID_ARG, "fa_fwd_bwd_host: problem too large");
  return FA_OK;
}

}  // namespace
}  // namespace fa

using namespace fa;

extern "C" {

size_t fa_fwd_bwd_host_workspace_size(int B, int H, int Hkv, int N, int d, fa_dtype dtype, int chunk) {
  if (check_args(B, H, Hkv, N, d, dtype, chunk) != FA_OK) return 0;
  const int units = B * Hkv;
  if (units == 0 || N == 0) return 0;
  const Slot s = slot_layout(chunk_units(units, chunk), H / Hkv, N, d, dtype == FA_FP32 ? 4 : 2);
  return 2 * s.total;
}

fa_status fa_fwd_bwd_host(const void* Q, const void* K, const void* V, const void* dO, void* O, float* L, void* dQ,
                          void* dK, void* dV, void* workspace, size_t workspace_bytes, int B, int H, int Hkv, int N,
                          int d, float scale, int causal, fa_dtype dtype, int chunk, void* stream) {
  fa_status st = check_args(B, H, Hkv, N, d, dtype, chunk);
  if (st != FA_OK) return st;
  const int units = B * Hkv, g = H / Hkv;
  if (units == 0 || N == 0) return FA_OK;
  const void* host[9] = {Q, K, V, dO, O, L, dQ, dK, dV};
  for (int i = 0; i < 9; ++i)
    if (!host[i]) return (fa_status)set_last_error(FA_ERR_INVALID_ARG, "fa_fwd_bwd_host: host pointer %d is null", i);
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)) != 0)
    return (fa_status)set_last_error(FA_ERR_INVALID_ARG, "fa_fwd_bwd_host: workspace must be 256-byte aligned");
  const int eb = dtype == FA_FP32 ? 4 : 2;
  const int cu = chunk_units(units, chunk);
  const Slot s = slot_layout(cu, g, N, d, eb);
  if (workspace_bytes < 2 * s.total)
    return (fa_status)set_last_error(FA_ERR_INVALID_ARG, "fa_fwd_bwd_host: workspace of %zu bytes < %zu required",
                                     workspace_bytes, 2 * s.total);
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices)
    return (fa_status)set_last_error(FA_ERR_UNSUPPORTED, "fa_fwd_bwd_host: device index %d out of range", dev);
  std::lock_guard<std::mutex> lk(g_pipe_mu[dev]);
  Pipe& p = g_pipe[dev];
  if ((st = pipe_init(p)) != FA_OK) return st;
  cudaStream_t user = static_cast<cudaStream_t>(stream);

  // after earlier work on the caller's stream and the previous call on these streams
  e = cudaEventRecord(p.start, user);
  for (cudaStream_t t : {p.in, p.comp, p.out}) {
    if (e == cudaSuccess) e = cudaStreamWaitEvent(t, p.start, 0);
    if (e == cudaSuccess && p.used) e = cudaStreamWaitEvent(t, p.fin, 0);
  }
  if (e != cudaSuccess) return cuda_fail(e, "ordering after the caller's stream");

  const size_t uq = (size_t)g * N * d * eb, uk = (size_t)N * d * eb, ul = (size_t)g * N * 4;  // bytes per unit
  auto hp = [](const void* base, size_t off) { return static_cast<const uint8_t*>(base) + off; };
  auto hw = [](void* base, size_t off) { return static_cast<uint8_t*>(base) + off; };
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int c = 0;
  for (int u0 = 0; u0 < units && st == FA_OK && e == cudaSuccess; u0 += cu, ++c) {
    const int nu = std::min(cu, units - u0);
    const int slot = c & 1;
    uint8_t* b = ws + slot * s.total;
    const size_t oq = (size_t)u0 * uq, ok_ = (size_t)u0 * uk, ol = (size_t)u0 * ul;
    const size_t nq = (size_t)nu * uq, nk = (size_t)nu * uk, nl = (size_t)nu * ul;
    // in: the slot's inputs were last read by chunk c - 2's computation
    if (c >= 2) e = cudaStreamWaitEvent(p.in, p.comp_done[slot], 0);
    if (e == cudaSuccess) e = cudaMemcpyAsync(b + s.q, hp(Q, oq), nq, cudaMemcpyHostToDevice, p.in);
    if (e == cudaSuccess) e = cudaMemcpyAsync(b + s.k, hp(K, ok_), nk, cudaMemcpyHostToDevice, p.in);
    if (e == cudaSuccess) e = cudaMemcpyAsync(b + s.v, hp(V, ok_), nk, cudaMemcpyHostToDevice, p.in);
    if (e == cudaSuccess) e = cudaMemcpyAsync(b + s.dout, hp(dO, oq), nq, cudaMemcpyHostToDevice, p.in);
    if (e == cudaSuccess) e = cudaEventRecord(p.in_ready[slot], p.in);
    // compute: the slot's outputs were last read by chunk c - 2's copy out
    if (e == cudaSuccess) e = cudaStreamWaitEvent(p.comp, p.in_ready[slot], 0);
    if (e == cudaSuccess && c >= 2) e = cudaStreamWaitEvent(p.comp, p.out_done[slot], 0);
    if (e != cudaSuccess) break;
    float* lse = reinterpret_cast<float*>(b + s.lse);
    st = fa_fwd_gqa(b + s.q, b + s.k, b + s.v, b + s.o, lse, 1, nu * g, nu, N, d, scale, causal, dtype, p.comp);
    if (st == FA_OK)
      st = fa_bwd_gqa(b + s.q, b + s.k, b + s.v, b + s.o, b + s.dout, lse, b + s.dq, b + s.dk, b + s.dv, b + s.ws,
                      s.ws_bytes, 1, nu * g, nu, N, d, scale, causal, dtype, p.comp);
    if (st != FA_OK) break;
    e = cudaEventRecord(p.comp_done[slot], p.comp);
    // out
    if (e == cudaSuccess) e = cudaStreamWaitEvent(p.out, p.comp_done[slot], 0);
    if (e == cudaSuccess) e = cudaMemcpyAsync(hw(O, oq), b + s.o, nq, cudaMemcpyDeviceToHost, p.out);
    if (e == cudaSuccess) e = cudaMemcpyAsync(hw(L, ol), b + s.lse, nl, cudaMemcpyDeviceToHost, p.out);
    if (e == cudaSuccess) e = cudaMemcpyAsync(hw(dQ, oq), b + s.dq, nq, cudaMemcpyDeviceToHost, p.out);
    if (e == cudaSuccess) e = cudaMemcpyAsync(hw(dK, ok_), b + s.dk, nk, cudaMemcpyDeviceToHost, p.out);
    if (e == cudaSuccess) e = cudaMemcpyAsync(hw(dV, ok_), b + s.dv, nk, cudaMemcpyDeviceToHost, p.out);
    if (e == cudaSuccess) e = cudaEventRecord(p.out_done[slot], p.out);
  }
  // whatever was enqueued, the caller's stream (and the next call) continue only after all of it
  cudaError_t e2 = cudaEventRecord(p.in_end, p.in);
  if (e2 == cudaSuccess) e2 = cudaEventRecord(p.comp_end, p.comp);
  if (e2 == cudaSuccess) e2 = cudaStreamWaitEvent(p.out, p.in_end, 0);
  if (e2 == cudaSuccess) e2 = cudaStreamWaitEvent(p.out, p.comp_end, 0);
  if (e2 == cudaSuccess) e2 = cudaEventRecord(p.fin, p.out);
  if (e2 == cudaSuccess) e2 = cudaStreamWaitEvent(user, p.fin, 0);
  if (e2 == cudaSuccess) p.used = true;
  if (st != FA_OK) return st;
  if (e != cudaSuccess) return cuda_fail(e, "enqueueing a chunk");
  if (e2 != cudaSuccess) return cuda_fail(e2, "ordering the caller's stream after the pipeline");
  return FA_OK;
}

}  // extern "C"
