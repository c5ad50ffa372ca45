"""Thin Python binding of the C ABI in ``include/fa.h`` (argument marshalling only).

Every entry point keeps the C name and takes torch CUDA tensors in place of
device pointers; shapes come from the tensors.  Nothing here computes: each
call checks the tensors, hands their pointers to ``libfa_gb300.so`` and turns a
non-OK status into ``FAError``.  If the library was not built the first call
raises: there is no fallback path.
"""

from __future__ import annotations

import ctypes
import os
import threading
import warnings

import torch

__all__ = [
    "FAError", "library_path", "load_library", "DTYPE_CODES",
    "fa_fwd", "fa_bwd", "fa_bwd_workspace_size", "fa_bwd_preprocess", "fa_bwd_main", "fa_bwd_dq_convert",
    "fa_check_device_error", "fa_tile_counter", "fa_uses_tensor_cores", "fa_status_string",
    "fa_last_error_message", "fa_bwd_noalloc", "fa_fwd_gqa", "fa_bwd_gqa", "fa_decode", "fa_decode_workspace_size",
    "fa_quantize_fp8", "fa_fwd_fp8", "fa_fwd_fp8_gqa", "fa_fwd_masked", "fa_bwd_masked",
    "fa_selftest_bounded_wait", "fa_fwd_bwd_host", "fa_fwd_bwd_host_workspace_size",
    "attention_forward", "attention_backward", "attention_decode",
    "attention_forward_fp8", "quantize_fp8", "EXPORTED_SYMBOLS", "NOALLOC_SCRATCH_BYTES",
    "fa_sm_clock_sample",
]

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_FILE = "libfa_gb300.so"

FA_OK = 0
NOALLOC_SCRATCH_BYTES = 64 << 20  # FA_BWD_NOALLOC_SCRATCH_BYTES in include/fa.h
DTYPE_CODES = {torch.bfloat16: 0, torch.float16: 1, torch.float32: 2}
EXPORTED_SYMBOLS = (
    "fa_fwd", "fa_bwd_workspace_size", "fa_bwd", "fa_bwd_preprocess", "fa_bwd_main", "fa_bwd_dq_convert",
    "fa_check_device_error", "fa_tile_counter", "fa_uses_tensor_cores", "fa_status_string",
    "fa_last_error_message", "fa_bwd_noalloc", "fa_fwd_gqa", "fa_bwd_gqa", "fa_decode", "fa_decode_workspace_size",
    "fa_quantize_fp8", "fa_fwd_fp8", "fa_fwd_fp8_gqa", "fa_fwd_masked", "fa_bwd_masked",
    "fa_selftest_bounded_wait", "fa_fwd_bwd_host", "fa_fwd_bwd_host_workspace_size", "fa_sm_clock_sample",
    "fa_debug_build", "fa_selftest_debug_check",
)

_lib = None
_lock = threading.Lock()


class FAError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{message} (status {status})")
        self.status = status


def library_path() -> str:
    return os.path.join(HERE, LIB_FILE)


def load_library(path=None):
    """Load ``libfa_gb300.so`` (built by ``exact_tiled_attention_07_gb300.build``); raises if absent.

    With ``path``, load that build of the library instead (for instance the FA_DEBUG build,
    ``build.build(debug=True)``) and make it the one every entry point here calls.
    """
    global _lib
    if path is None and _lib is not None:
        return _lib
    with _lock:
        if path is None and _lib is not None:
            return _lib
        path = path or library_path()
        if not os.path.exists(path):
            raise RuntimeError(f"the CUDA library {path} is not built; run __graft_entry__.build() first")
        lib = ctypes.CDLL(path)
        vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        lib.fa_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, i, i, vp]
        lib.fa_bwd_workspace_size.argtypes = [i, i, i, i]
        lib.fa_bwd_workspace_size.restype = sz
        lib.fa_bwd.argtypes = [vp] * 10 + [sz, i, i, i, i, f, i, i, vp]
        lib.fa_bwd_preprocess.argtypes = [vp, vp, vp, vp, sz, i, i, i, i, i, vp]
        lib.fa_bwd_main.argtypes = [vp] * 7 + [sz, i, i, i, i, f, i, i, vp]
        lib.fa_bwd_dq_convert.argtypes = [vp, sz, vp, i, i, i, i, f, i, vp]
        lib.fa_bwd_noalloc.argtypes = [vp] * 9 + [i, i, i, i, f, i, i, vp]
        lib.fa_fwd_gqa.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, i, vp]
        lib.fa_bwd_gqa.argtypes = [vp] * 10 + [sz, i, i, i, i, i, f, i, i, vp]
        lib.fa_decode_workspace_size.argtypes = [i] * 7
        lib.fa_decode_workspace_size.restype = sz
        lib.fa_decode.argtypes = [vp] * 5 + [i] * 6 + [f, i, i, vp, sz, vp]
        lib.fa_quantize_fp8.argtypes = [vp, vp, vp, i, i, i, i, i, vp]
        lib.fa_fwd_masked.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, i, vp, i, i, vp]
        lib.fa_bwd_masked.argtypes = [vp] * 10 + [sz, i, i, i, i, i, f, i, i, vp, i, i, vp]
        lib.fa_fwd_fp8.argtypes = [vp] * 8 + [i, i, i, i, f, i, i, vp]
        lib.fa_fwd_fp8_gqa.argtypes = [vp] * 8 + [i, i, i, i, i, f, i, i, vp]
        lib.fa_selftest_bounded_wait.argtypes = [i, i, vp]
        lib.fa_fwd_bwd_host_workspace_size.argtypes = [i, i, i, i, i, i, i]
        lib.fa_fwd_bwd_host_workspace_size.restype = sz
        lib.fa_fwd_bwd_host.argtypes = [vp] * 10 + [sz, i, i, i, i, i, f, i, i, i, vp]
        lib.fa_check_device_error.argtypes = [vp]
        lib.fa_sm_clock_sample.argtypes = [vp, i, vp]
        lib.fa_debug_build.argtypes = []
        lib.fa_debug_build.restype = ctypes.c_int
        lib.fa_selftest_debug_check.argtypes = [i, i, vp]
        lib.fa_tile_counter.argtypes = [vp, ctypes.POINTER(ctypes.c_ulonglong), i]
        lib.fa_uses_tensor_cores.argtypes = [i, i, i]
        lib.fa_status_string.argtypes = [i]
        lib.fa_status_string.restype = ctypes.c_char_p
        lib.fa_last_error_message.argtypes = []
        lib.fa_last_error_message.restype = ctypes.c_char_p
        for name in ("fa_fwd", "fa_bwd", "fa_fwd_gqa", "fa_bwd_gqa", "fa_decode", "fa_quantize_fp8", "fa_fwd_fp8",
                     "fa_fwd_fp8_gqa",
                     "fa_fwd_masked", "fa_bwd_masked", "fa_selftest_bounded_wait", "fa_fwd_bwd_host",
                     "fa_bwd_noalloc", "fa_bwd_preprocess",
                     "fa_bwd_main", "fa_bwd_dq_convert",
                     "fa_check_device_error", "fa_tile_counter", "fa_uses_tensor_cores", "fa_sm_clock_sample",
                     "fa_selftest_debug_check"):
            getattr(lib, name).restype = ctypes.c_int
        _lib = lib
        return lib


def _check(status: int):
    if status != FA_OK:
        lib = load_library()
        msg = lib.fa_last_error_message().decode() or lib.fa_status_string(status).decode()
        raise FAError(status, msg)


def _stream(stream):
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _p(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _shape4(t):
    if t.dim() != 4:
        raise ValueError(f"expected a [B, H, N, d] tensor, got shape {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous [B, H, N, d]")
    return tuple(int(s) for s in t.shape)


def _dt(t):
    try:
        return DTYPE_CODES[t.dtype]
    except KeyError:
        raise ValueError(f"unsupported dtype {t.dtype}") from None


def _on_device(*ts):
    """Every tensor given (None is skipped) is a contiguous CUDA tensor on the current device:
    the library takes raw device pointers and launches on the current device, so a host tensor
    or one on another GPU would hand the kernels an address they cannot use."""
    dev = None
    for t in ts:
        if t is None:
            continue
        if not t.is_cuda:
            raise ValueError("device arguments must be CUDA tensors (the library takes device pointers)")
        if not t.is_contiguous():
            raise ValueError("device arguments must be contiguous")
        if dev is None:
            dev, cur = t.device.index, torch.cuda.current_device()
            if dev != cur:
                raise ValueError(f"tensors are on cuda:{dev} but the current device is cuda:{cur}; "
                                 f"call within torch.cuda.device({dev})")
        elif t.device.index != dev:
            raise ValueError("all device arguments must be on one GPU")


def _rows(L, n, what="L"):
    """L (or another per-row vector) is an fp32 tensor of n elements."""
    if L.dtype != torch.float32 or L.numel() != n:
        raise ValueError(f"{what} must be an fp32 tensor of {n} elements")


def _same(ref, *ts):
    for t in ts:
        if t.shape != ref.shape or t.dtype != ref.dtype or t.device != ref.device or not t.is_contiguous():
            raise ValueError("Q, K, V, O, dO, dQ, dK, dV must share shape, dtype and device and be contiguous")


def fa_fwd(Q, K, V, O, L, scale, causal, stream=None):
    B, H, N, d = _shape4(Q)
    _on_device(Q, K, V, O, L)
    _same(Q, K, V, O)
    if L.dtype != torch.float32 or L.numel() != B * H * N or not L.is_contiguous():
        raise ValueError("L must be a contiguous fp32 tensor of B*H*N elements")
    _check(load_library().fa_fwd(_p(Q), _p(K), _p(V), _p(O), _p(L), B, H, N, d, float(scale), int(bool(causal)),
                                 _dt(Q), _stream(stream)))


def _kv_heads(Q, K, V, *kv_like):
    """Key/value head count of K (grouped-query attention) after checking the shapes agree."""
    B, H, N, d = _shape4(Q)
    Bk, Hkv, Nk, dk = _shape4(K)
    if (Bk, Nk, dk) != (B, N, d) or Hkv < 1 or H % Hkv:
        raise ValueError("K must be [B, Hkv, N, d] with H a multiple of Hkv")
    for t in (V,) + kv_like:
        if t.shape != K.shape or t.dtype != Q.dtype or t.device != Q.device or not t.is_contiguous():
            raise ValueError("K, V (and dK, dV) must share shape, dtype and device and be contiguous")
    return Hkv


def fa_fwd_gqa(Q, K, V, O, L, scale, causal, stream=None):
    B, H, N, d = _shape4(Q)
    _on_device(Q, K, V, O, L)
    Hkv = _kv_heads(Q, K, V)
    _same(Q, O)
    if L.dtype != torch.float32 or L.numel() != B * H * N or not L.is_contiguous():
        raise ValueError("L must be a contiguous fp32 tensor of B*H*N elements")
    _check(load_library().fa_fwd_gqa(_p(Q), _p(K), _p(V), _p(O), _p(L), B, H, Hkv, N, d, float(scale),
                                     int(bool(causal)), _dt(Q), _stream(stream)))


def fa_bwd_gqa(Q, K, V, O, dO, L, dQ, dK, dV, workspace, scale, causal, stream=None):
    B, H, N, d = _shape4(Q)
    _on_device(Q, K, V, O, dO, L, dQ, dK, dV, workspace)
    Hkv = _kv_heads(Q, K, V, dK, dV)
    _same(Q, O, dO, dQ)
    _rows(L, B * H * N)
    _check(load_library().fa_bwd_gqa(_p(Q), _p(K), _p(V), _p(O), _p(dO), _p(L), _p(dQ), _p(dK), _p(dV),
                                     _p(workspace), workspace.numel() * workspace.element_size(), B, H, Hkv, N, d,
                                     float(scale), int(bool(causal)), _dt(Q), _stream(stream)))


def fa_bwd_workspace_size(B, H, N, d) -> int:
    return int(load_library().fa_bwd_workspace_size(B, H, N, d))


def fa_bwd(Q, K, V, O, dO, L, dQ, dK, dV, workspace, scale, causal, stream=None):
    B, H, N, d = _shape4(Q)
    _on_device(Q, K, V, O, dO, L, dQ, dK, dV, workspace)
    _same(Q, K, V, O, dO, dQ, dK, dV)
    _rows(L, B * H * N)
    _check(load_library().fa_bwd(_p(Q), _p(K), _p(V), _p(O), _p(dO), _p(L), _p(dQ), _p(dK), _p(dV), _p(workspace),
                                 workspace.numel() * workspace.element_size(), B, H, N, d, float(scale),
                                 int(bool(causal)), _dt(Q), _stream(stream)))


def fa_bwd_preprocess(O, dO, L, workspace, stream=None):
    B, H, N, d = _shape4(O)
    _on_device(O, dO, L, workspace)
    _same(O, dO)
    _rows(L, B * H * N)
    _check(load_library().fa_bwd_preprocess(_p(O), _p(dO), _p(L), _p(workspace),
                                            workspace.numel() * workspace.element_size(), B, H, N, d, _dt(O),
                                            _stream(stream)))


def fa_bwd_main(Q, K, V, dO, dK, dV, workspace, scale, causal, stream=None):
    B, H, N, d = _shape4(Q)
    _on_device(Q, K, V, dO, dK, dV, workspace)
    _same(Q, K, V, dO, dK, dV)
    _check(load_library().fa_bwd_main(_p(Q), _p(K), _p(V), _p(dO), _p(dK), _p(dV), _p(workspace),
                                      workspace.numel() * workspace.element_size(), B, H, N, d, float(scale),
                                      int(bool(causal)), _dt(Q), _stream(stream)))


def fa_bwd_dq_convert(workspace, dQ, scale, stream=None):
    B, H, N, d = _shape4(dQ)
    _on_device(workspace, dQ)
    _check(load_library().fa_bwd_dq_convert(_p(workspace), workspace.numel() * workspace.element_size(), _p(dQ),
                                            B, H, N, d, float(scale), _dt(dQ), _stream(stream)))


def fa_bwd_noalloc(Q, K, V, O, dO, L, dQ, dK, dV, scale, causal, stream=None):
    """fa_bwd with the library's static device scratch instead of a workspace (no allocation)."""
    B, H, N, d = _shape4(Q)
    _on_device(Q, K, V, O, dO, L, dQ, dK, dV)
    _same(Q, K, V, O, dO, dQ, dK, dV)
    _rows(L, B * H * N)
    _check(load_library().fa_bwd_noalloc(_p(Q), _p(K), _p(V), _p(O), _p(dO), _p(L), _p(dQ), _p(dK), _p(dV), B, H, N,
                                         d, float(scale), int(bool(causal)), _dt(Q), _stream(stream)))


def fa_fwd_bwd_host_workspace_size(B, H, Hkv, N, d, dtype, chunk=0) -> int:
    return int(load_library().fa_fwd_bwd_host_workspace_size(B, H, Hkv, N, d, DTYPE_CODES[dtype], int(chunk)))


def fa_fwd_bwd_host(Q, K, V, dO, O, L, dQ, dK, dV, workspace, scale, causal, chunk=0, stream=None):
    """Forward + backward with CPU tensors in and out (page-locked for the copies to overlap) and
    a device workspace of fa_fwd_bwd_host_workspace_size bytes."""
    B, H, N, d = _shape4(Q)
    Bk, Hkv, Nk, dk = _shape4(K)
    if (Bk, Nk, dk) != (B, N, d) or Hkv < 1 or H % Hkv:
        raise ValueError("K must be [B, Hkv, N, d] with H a multiple of Hkv")
    for t in (Q, K, V, dO, O, L, dQ, dK, dV):
        if t.device.type != "cpu" or not t.is_contiguous():
            raise ValueError("fa_fwd_bwd_host takes contiguous host (CPU) tensors")
    for t in (V, dK, dV):
        if t.shape != K.shape or t.dtype != Q.dtype:
            raise ValueError("V, dK, dV must be [B, Hkv, N, d] of Q's dtype")
    for t in (dO, O, dQ):
        if t.shape != Q.shape or t.dtype != Q.dtype:
            raise ValueError("dO, O, dQ must be [B, H, N, d] of Q's dtype")
    if L.dtype != torch.float32 or L.numel() != B * H * N:
        raise ValueError("L must be an fp32 tensor of B*H*N elements")
    if workspace.device.type != "cuda":
        raise ValueError("the workspace is device memory")
    _on_device(workspace)
    _check(load_library().fa_fwd_bwd_host(_p(Q), _p(K), _p(V), _p(dO), _p(O), _p(L), _p(dQ), _p(dK), _p(dV),
                                          _p(workspace), workspace.numel() * workspace.element_size(), B, H, Hkv, N,
                                          d, float(scale), int(bool(causal)), _dt(Q), int(chunk), _stream(stream)))


def fa_decode_workspace_size(B, H, Hkv, Nq, Nk, d, splits=0) -> int:
    return int(load_library().fa_decode_workspace_size(B, H, Hkv, Nq, Nk, d, int(splits)))


def fa_decode(Q, K, V, O, L, scale, splits=0, workspace=None, stream=None):
    """Decode: Q, O [B, H, Nq, d] against the cache K, V [B, Hkv, Nk, d]; L [B, H, Nq]."""
    B, H, Nq, d = _shape4(Q)
    Bk, Hkv, Nk, dk = _shape4(K)
    _on_device(Q, K, V, O, L, workspace)
    if (Bk, dk) != (B, d) or V.shape != K.shape or V.dtype != Q.dtype or K.dtype != Q.dtype or not V.is_contiguous():
        raise ValueError("K, V must be [B, Hkv, Nk, d] of Q's dtype")
    _same(Q, O)
    if L.dtype != torch.float32 or L.numel() != B * H * Nq or not L.is_contiguous():
        raise ValueError("L must be a contiguous fp32 tensor of B*H*Nq elements")
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load_library().fa_decode(_p(Q), _p(K), _p(V), _p(O), _p(L), B, H, Hkv, Nq, Nk, d, float(scale), int(splits),
                                    _dt(Q), _p(workspace), nbytes, _stream(stream)))


def fa_quantize_fp8(X, X8, scales, stream=None):
    """Block quantisation of X [B, H, N, d] to E4M3 codes X8 (uint8, same shape) and
    scales [B, H, ceil(N / 128)] fp32."""
    B, H, N, d = _shape4(X)
    _on_device(X, X8, scales)
    if X8.dtype != torch.uint8 or tuple(X8.shape) != (B, H, N, d) or not X8.is_contiguous():
        raise ValueError("X8 must be a contiguous uint8 tensor of X's shape")
    nb = (N + 127) // 128
    if scales.dtype != torch.float32 or scales.numel() != B * H * nb or not scales.is_contiguous():
        raise ValueError(f"scales must be a contiguous fp32 tensor of B*H*ceil(N/128) = {B * H * nb} elements")
    _check(load_library().fa_quantize_fp8(_p(X), _p(X8), _p(scales), B, H, N, d, _dt(X), _stream(stream)))


def fa_fwd_fp8(Q8, K8, V8, q_scales, k_scales, v_scales, O, L, scale, causal, stream=None):
    """Forward on E4M3 codes with block scales; O [B, H, N, d] bf16 or fp16, L [B, H, N] fp32.
    K8, V8 (and their scales) may have fewer heads than Q8 (grouped-query: fa_fwd_fp8_gqa)."""
    B, H, N, d = _shape4(Q8)
    Hkv = _shape4(K8)[1]
    _on_device(Q8, K8, V8, q_scales, k_scales, v_scales, O, L)
    nb = (N + 127) // 128
    for t, heads in ((Q8, H), (K8, Hkv), (V8, Hkv)):
        if t.dtype != torch.uint8 or tuple(t.shape) != (B, heads, N, d) or not t.is_contiguous():
            raise ValueError("Q8 [B, H, N, d] and K8, V8 [B, Hkv, N, d] must be contiguous uint8 tensors")
    if Hkv < 1 or H % Hkv:
        raise ValueError("H must be a multiple of the key/value heads Hkv")
    for t, heads in ((q_scales, H), (k_scales, Hkv), (v_scales, Hkv)):
        if t.dtype != torch.float32 or t.numel() != B * heads * nb or not t.is_contiguous():
            raise ValueError("block scales must be contiguous fp32 tensors of B*heads*ceil(N/128) elements")
    if tuple(O.shape) != (B, H, N, d) or not O.is_contiguous():
        raise ValueError("O must be a contiguous [B, H, N, d] tensor")
    if L.dtype != torch.float32 or L.numel() != B * H * N or not L.is_contiguous():
        raise ValueError("L must be a contiguous fp32 tensor of B*H*N elements")
    if Hkv != H:
        _check(load_library().fa_fwd_fp8_gqa(_p(Q8), _p(K8), _p(V8), _p(q_scales), _p(k_scales), _p(v_scales), _p(O),
                                             _p(L), B, H, Hkv, N, d, float(scale), int(bool(causal)), _dt(O),
                                             _stream(stream)))
        return
    _check(load_library().fa_fwd_fp8(_p(Q8), _p(K8), _p(V8), _p(q_scales), _p(k_scales), _p(v_scales), _p(O), _p(L),
                                     B, H, N, d, float(scale), int(bool(causal)), _dt(O), _stream(stream)))


def fa_fwd_fp8_gqa(Q8, K8, V8, q_scales, k_scales, v_scales, O, L, scale, causal, stream=None):
    """fa_fwd_fp8 with K8, V8 of Hkv heads (H a multiple of Hkv); the same checks."""
    fa_fwd_fp8(Q8, K8, V8, q_scales, k_scales, v_scales, O, L, scale, causal, stream)


def _mask_args(block_mask, H):
    """(pointer, mask_heads) of a uint8 block mask [nb, nb] (shared) or [H, nb, nb] (per head)."""
    if block_mask is None:
        return ctypes.c_void_p(0), 0
    if block_mask.dtype != torch.uint8 or not block_mask.is_contiguous() or not block_mask.is_cuda:
        raise ValueError("block_mask must be a contiguous uint8 CUDA tensor")
    heads = 1 if block_mask.dim() == 2 else block_mask.shape[0]
    return _p(block_mask), heads


def fa_fwd_masked(Q, K, V, O, L, scale, causal, window=0, block_mask=None, stream=None):
    """Forward with a sliding window and/or a block mask over 128 x 128 score blocks."""
    B, H, N, d = _shape4(Q)
    _on_device(Q, K, V, O, L, block_mask)
    Hkv = _kv_heads(Q, K, V)
    _same(Q, O)
    _rows(L, B * H * N)
    mp, mh = _mask_args(block_mask, H)
    _check(load_library().fa_fwd_masked(_p(Q), _p(K), _p(V), _p(O), _p(L), B, H, Hkv, N, d, float(scale),
                                        int(bool(causal)), int(window), mp, mh, _dt(Q), _stream(stream)))


def fa_bwd_masked(Q, K, V, O, dO, L, dQ, dK, dV, workspace, scale, causal, window=0, block_mask=None, stream=None):
    """Backward of fa_fwd_masked (same mask)."""
    B, H, N, d = _shape4(Q)
    _on_device(Q, K, V, O, dO, L, dQ, dK, dV, workspace, block_mask)
    Hkv = _kv_heads(Q, K, V, dK, dV)
    _same(Q, O, dO, dQ)
    _rows(L, B * H * N)
    mp, mh = _mask_args(block_mask, H)
    nbytes = workspace.numel() * workspace.element_size()
    _check(load_library().fa_bwd_masked(_p(Q), _p(K), _p(V), _p(O), _p(dO), _p(L), _p(dQ), _p(dK), _p(dV),
                                        _p(workspace), nbytes, B, H, Hkv, N, d, float(scale), int(bool(causal)),
                                        int(window), mp, mh, _dt(Q), _stream(stream)))


def fa_selftest_bounded_wait(timeout_ms=20, arrive=False, stream=None):
    """Launch the bounded-wait self-test (see include/fa.h); read the outcome with fa_check_device_error."""
    _check(load_library().fa_selftest_bounded_wait(int(timeout_ms), int(bool(arrive)), _stream(stream)))


def fa_sm_clock_sample(out, stream=None):
    """Enqueue one reading of every SM's cycle counter and the global timer into ``out``, a CUDA
    uint64 (or int64) tensor of 3 x blocks elements, blocks <= the SM count (see include/fa.h)."""
    _on_device(out)
    if out.element_size() != 8 or out.numel() % 3 != 0:
        raise ValueError("out must hold 3 x blocks 64-bit words")
    _check(load_library().fa_sm_clock_sample(_p(out), out.numel() // 3, _stream(stream)))


def fa_debug_build() -> bool:
    """Whether the loaded library was built with FA_DEBUG (device-side index checks)."""
    return bool(load_library().fa_debug_build())


def fa_selftest_debug_check(index, limit, stream=None):
    """Launch one device index check of index against [0, limit) (debug builds; see include/fa.h)."""
    _check(load_library().fa_selftest_debug_check(int(index), int(limit), _stream(stream)))


def fa_check_device_error(stream=None):
    _check(load_library().fa_check_device_error(_stream(stream)))


def fa_tile_counter(stream=None, reset=False) -> int:
    v = ctypes.c_ulonglong(0)
    _check(load_library().fa_tile_counter(_stream(stream), ctypes.byref(v), int(bool(reset))))
    return int(v.value)


def fa_uses_tensor_cores(pass_: str, dtype, d: int) -> bool:
    code = DTYPE_CODES[dtype] if isinstance(dtype, torch.dtype) else int(dtype)
    return bool(load_library().fa_uses_tensor_cores(0 if pass_ == "fwd" else 1, code, int(d)))


def fa_status_string(status: int) -> str:
    return load_library().fa_status_string(int(status)).decode()


def fa_last_error_message() -> str:
    return load_library().fa_last_error_message().decode()


# ---------------------------------------------------------------------------
# conveniences: allocate outputs with torch, then call the entry points above
# ---------------------------------------------------------------------------


def _warn_cuda_core(pass_, t, d):
    """A 16-bit pass with no tensor-core kernel runs on the CUDA-core kernels: say so."""
    if t.dtype != torch.float32 and not fa_uses_tensor_cores(pass_, t.dtype, d):
        warnings.warn(f"{t.dtype} {'forward' if pass_ == 'fwd' else 'backward'} at d={d} runs on the CUDA-core "
                      f"kernels (fp32 arithmetic): no tensor-core kernel for this head dimension", stacklevel=3)


def attention_forward(q, k, v, causal=False, scale=None, stream=None, window=0, block_mask=None):
    """O, L = fa_fwd(q, k, v) (fa_fwd_gqa when k, v have fewer heads than q; fa_fwd_masked with a
    window or a block mask); outputs on q's device."""
    B, H, N, d = _shape4(q)
    _warn_cuda_core("fwd", q, d)
    scale = d ** -0.5 if scale is None else scale
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    if window or block_mask is not None:
        fa_fwd_masked(q, k, v, o, lse, scale, causal, window, block_mask, stream)
    elif k.shape[1] != H:
        fa_fwd_gqa(q, k, v, o, lse, scale, causal, stream)
    else:
        fa_fwd(q, k, v, o, lse, scale, causal, stream)
    return o, lse


def attention_backward(q, k, v, o, do, lse, causal=False, scale=None, workspace=None, stream=None, window=0,
                       block_mask=None):
    """dQ, dK, dV = fa_bwd(...) (fa_bwd_masked with a window or a block mask); outputs (and
    workspace, unless given) allocated with torch."""
    B, H, N, d = _shape4(q)
    _warn_cuda_core("bwd", q, d)
    scale = d ** -0.5 if scale is None else scale
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    if workspace is None:
        nbytes = fa_bwd_workspace_size(B, H, N, d)
        workspace = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=q.device)
    if window or block_mask is not None:
        fa_bwd_masked(q, k, v, o, do, lse, dq, dk, dv, workspace, scale, causal, window, block_mask, stream)
    elif k.shape[1] != H:
        fa_bwd_gqa(q, k, v, o, do, lse, dq, dk, dv, workspace, scale, causal, stream)
    else:
        fa_bwd(q, k, v, o, do, lse, dq, dk, dv, workspace, scale, causal, stream)
    return dq, dk, dv


def attention_decode(q, k, v, scale=None, splits=0, stream=None):
    """O, L = fa_decode(q, k, v) for q [B, H, Nq, d] over the cache k, v [B, Hkv, Nk, d]."""
    B, H, Nq, d = _shape4(q)
    _, Hkv, Nk, _ = _shape4(k)
    scale = d ** -0.5 if scale is None else scale
    o = torch.empty_like(q)
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    nbytes = fa_decode_workspace_size(B, H, Hkv, Nq, Nk, d, splits)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=q.device) if nbytes else None
    fa_decode(q, k, v, o, lse, scale, splits, ws, stream)
    return o, lse


def quantize_fp8(x, stream=None):
    """(codes, scales) = block quantisation of x [B, H, N, d] (one scale per 128 rows of a head)."""
    B, H, N, d = _shape4(x)
    x8 = torch.empty((B, H, N, d), dtype=torch.uint8, device=x.device)
    sc = torch.empty((B, H, (N + 127) // 128), dtype=torch.float32, device=x.device)
    fa_quantize_fp8(x, x8, sc, stream)
    return x8, sc


def attention_forward_fp8(q8, k8, v8, q_scales, k_scales, v_scales, scale=None, causal=False,
                          out_dtype=torch.bfloat16, stream=None):
    """O, L = fa_fwd_fp8(...) on E4M3 codes and their block scales."""
    B, H, N, d = _shape4(q8)
    scale = d ** -0.5 if scale is None else scale
    o = torch.empty((B, H, N, d), dtype=out_dtype, device=q8.device)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q8.device)
    fa_fwd_fp8(q8, k8, v8, q_scales, k_scales, v_scales, o, lse, scale, causal, stream)
    return o, lse
