"""The C-ABI library builds, loads and exports every declared symbol; host-side argument checks (no GPU)."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from exact_tiled_attention_07_gb300 import build as b

    path = b.build()
    assert os.path.exists(path)
    return ctypes.CDLL(path)


def _declared_symbols():
    txt = open(os.path.join(ROOT, "include", "fa.h")).read()
    return re.findall(r"FA_API\s+[\w\s\*]*?\b(fa_\w+)\s*\(", txt)


def test_header_declares_the_boundary():
    names = set(_declared_symbols())
    for required in ("fa_fwd", "fa_bwd", "fa_bwd_workspace_size", "fa_check_device_error", "fa_status_string"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_symbols():
        assert hasattr(lib, name), name


def test_binding_covers_every_symbol():
    from exact_tiled_attention_07_gb300 import binding

    assert set(binding.EXPORTED_SYMBOLS) == set(_declared_symbols())
    for name in _declared_symbols():
        assert callable(getattr(binding, name))


def test_noalloc_scratch_size_matches_the_header():
    # the binding's copy of FA_BWD_NOALLOC_SCRATCH_BYTES, which its size checks and tests use
    from exact_tiled_attention_07_gb300 import binding

    txt = open(os.path.join(ROOT, "include", "fa.h")).read()
    m = re.search(r"#define\s+FA_BWD_NOALLOC_SCRATCH_BYTES\s+\((\d+)ull\s*<<\s*(\d+)\)", txt)
    assert m, "FA_BWD_NOALLOC_SCRATCH_BYTES not found in include/fa.h"
    assert binding.NOALLOC_SCRATCH_BYTES == int(m.group(1)) << int(m.group(2))


def test_status_strings(lib):
    lib.fa_status_string.restype = ctypes.c_char_p
    assert lib.fa_status_string(0) == b"ok"
    assert b"timed out" in lib.fa_status_string(4)
    assert lib.fa_status_string(99) == b"unknown status"


def test_workspace_size_is_linear_in_n(lib):
    lib.fa_bwd_workspace_size.restype = ctypes.c_size_t
    ws = lambda b, h, n, d: lib.fa_bwd_workspace_size(b, h, n, d)
    # D + L*log2e + fp32 dQ accumulator over N rounded up to 128, then 256 bytes of queue
    # counters: nothing N x N
    assert ws(1, 1, 128, 64) == 128 * 4 * 66 + 256
    assert ws(2, 3, 129, 128) == 6 * 256 * 4 * 130 + 256
    assert ws(8, 16, 4096, 128) == 8 * 16 * 4096 * 4 * 130 + 256
    assert ws(1, 8, 65536, 64) < 65536 * 65536  # vs. one N x N byte matrix
    assert ws(1, 1, 16, 0) == 0 and ws(1, 1, 16, 300) == 0


def test_invalid_arguments_are_rejected_without_launching(lib):
    vp = ctypes.c_void_p
    lib.fa_fwd.argtypes = [vp, vp, vp, vp, vp, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                           ctypes.c_float, ctypes.c_int, ctypes.c_int, vp]
    lib.fa_last_error_message.restype = ctypes.c_char_p
    good = vp(0x10000)
    # empty problems succeed and launch nothing
    assert lib.fa_fwd(None, None, None, None, None, 0, 4, 128, 64, 0.125, 0, 0, None) == 0
    assert lib.fa_fwd(None, None, None, None, None, 2, 4, 0, 64, 0.125, 0, 0, None) == 0
    # null / misaligned pointers
    assert lib.fa_fwd(None, good, good, good, good, 1, 1, 128, 64, 0.125, 0, 0, None) == 1
    assert b"null" in lib.fa_last_error_message()
    assert lib.fa_fwd(vp(0x10008), good, good, good, good, 1, 1, 128, 64, 0.125, 0, 0, None) == 1
    assert b"aligned" in lib.fa_last_error_message()
    # sizes, dtype, head dim, scale
    assert lib.fa_fwd(good, good, good, good, good, -1, 1, 128, 64, 0.125, 0, 0, None) == 1
    assert lib.fa_fwd(good, good, good, good, good, 1, 1, 128, 512, 0.125, 0, 0, None) == 2
    assert lib.fa_fwd(good, good, good, good, good, 1, 1, 128, 64, 0.125, 0, 7, None) == 2
    assert lib.fa_fwd(good, good, good, good, good, 1, 1, 128, 64, float("nan"), 0, 0, None) == 1
    assert lib.fa_fwd(good, good, good, good, good, 1, 1, 128, 64, -1.0, 0, 0, None) == 1


def test_backward_workspace_too_small_is_rejected(lib):
    vp = ctypes.c_void_p
    lib.fa_bwd.argtypes = [vp] * 10 + [ctypes.c_size_t, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                       ctypes.c_float, ctypes.c_int, ctypes.c_int, vp]
    lib.fa_last_error_message.restype = ctypes.c_char_p
    g = vp(0x10000)
    st = lib.fa_bwd(g, g, g, g, g, g, g, g, g, g, 1024, 1, 1, 128, 64, 0.125, 0, 0, None)
    assert st == 1 and b"workspace" in lib.fa_last_error_message()


def test_kernel_selection(lib):
    lib.fa_uses_tensor_cores.argtypes = [ctypes.c_int] * 3
    for d in (64, 128, 256):
        assert lib.fa_uses_tensor_cores(0, 0, d) == 1  # bf16 forward
        assert lib.fa_uses_tensor_cores(0, 1, d) == 1  # fp16 forward
        assert lib.fa_uses_tensor_cores(0, 2, d) == 0  # fp32: CUDA cores
    assert lib.fa_uses_tensor_cores(1, 0, 128) == 1 and lib.fa_uses_tensor_cores(1, 0, 256) == 1
    assert lib.fa_uses_tensor_cores(1, 1, 96) == 0
    assert lib.fa_uses_tensor_cores(0, 0, 96) == 0


def test_oracle_is_not_imported_by_the_product():
    pkg = os.path.join(ROOT, "exact_tiled_attention_07_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                txt = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"^\s*(from|import)\s+oracle\b", txt, re.M), f
                assert "oracle/" not in txt, f


def test_gqa_head_counts_are_validated(lib):
    vp, i = ctypes.c_void_p, ctypes.c_int
    lib.fa_fwd_gqa.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, ctypes.c_float, i, i, vp]
    lib.fa_last_error_message.restype = ctypes.c_char_p
    g = vp(0x10000)
    assert lib.fa_fwd_gqa(g, g, g, g, g, 1, 4, 3, 128, 64, 0.125, 0, 0, None) == 1
    assert b"multiple" in lib.fa_last_error_message()
    assert lib.fa_fwd_gqa(g, g, g, g, g, 1, 4, 0, 128, 64, 0.125, 0, 0, None) == 1


def test_decode_workspace_size_host_rules(lib):
    lib.fa_decode_workspace_size.argtypes = [ctypes.c_int] * 7
    lib.fa_decode_workspace_size.restype = ctypes.c_size_t
    f = lib.fa_decode_workspace_size
    assert f(1, 8, 2, 1, 100, 128, 1) == 0  # one piece: no workspace
    assert f(2, 8, 2, 3, 1000, 64, 5) == 2 * 8 * 3 * 5 * 65 * 4
    assert f(1, 8, 3, 1, 100, 128, 4) == 0  # heads do not divide: invalid
    assert f(1, 8, 2, 1, 100, 96, 4) == 0  # unsupported head dim
    assert f(1, 8, 2, 1, 1 << 20, 128, 0) > 0  # long cache: split automatically


def test_mask_arguments_are_validated(lib):
    vp, i = ctypes.c_void_p, ctypes.c_int
    lib.fa_fwd_masked.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, ctypes.c_float, i, i, vp, i, i, vp]
    lib.fa_last_error_message.restype = ctypes.c_char_p
    g = vp(0x10000)
    # negative window; mask_heads without a mask; mask_heads neither 1 nor H
    assert lib.fa_fwd_masked(g, g, g, g, g, 1, 4, 4, 128, 64, 0.125, 1, -1, None, 0, 0, None) == 1
    assert lib.fa_fwd_masked(g, g, g, g, g, 1, 4, 4, 128, 64, 0.125, 1, 8, None, 1, 0, None) == 1
    assert lib.fa_fwd_masked(g, g, g, g, g, 1, 4, 4, 128, 64, 0.125, 0, 0, g, 3, 0, None) == 1
    assert b"mask_heads" in lib.fa_last_error_message()
    # masks run on the tensor-core kernels only: fp32 and odd head dims are unsupported
    assert lib.fa_fwd_masked(g, g, g, g, g, 1, 4, 4, 128, 64, 0.125, 1, 8, None, 0, 2, None) == 2
    assert lib.fa_fwd_masked(g, g, g, g, g, 1, 4, 4, 128, 96, 0.125, 1, 8, None, 0, 0, None) == 2


def test_selftest_timeout_range(lib):
    lib.fa_selftest_bounded_wait.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_void_p]
    assert lib.fa_selftest_bounded_wait(0, 0, None) == 1
    assert lib.fa_selftest_bounded_wait(5000, 0, None) == 1


def test_host_pipeline_workspace_size_host_rules(lib):
    f = lib.fa_fwd_bwd_host_workspace_size
    f.argtypes = [ctypes.c_int] * 7
    f.restype = ctypes.c_size_t
    bf16 = 0
    # invalid shapes, dtype or chunk: 0; nothing to do: 0
    assert f(1, 4, 3, 128, 64, bf16, 0) == 0
    assert f(1, 4, 2, 128, 0, bf16, 0) == 0
    assert f(1, 4, 2, 128, 64, 7, 0) == 0
    assert f(1, 4, 2, 128, 64, bf16, -1) == 0
    assert f(0, 4, 2, 128, 64, bf16, 0) == 0
    # two slots; one key/value head (2 query heads) of N = 128, d = 64, bf16 per slot:
    # Q, dO, O, dQ 2 x 16 KB each; K, V, dK, dV 16 KB each; L 1 KB; backward workspace
    one = f(1, 4, 2, 128, 64, bf16, 1)
    ws = lib.fa_bwd_workspace_size
    ws.argtypes = [ctypes.c_int] * 4
    ws.restype = ctypes.c_size_t
    assert one == 2 * (4 * 32768 + 4 * 16384 + 1024 + ws(1, 2, 128, 64))
    # chunks larger than the problem are clipped; the automatic choice is about eight chunks
    assert f(1, 4, 2, 128, 64, bf16, 5) == f(1, 4, 2, 128, 64, bf16, 2)
    assert f(8, 16, 16, 4096, 128, bf16, 0) == f(8, 16, 16, 4096, 128, bf16, 16)


def test_host_pipeline_rejects_null_host_pointers_before_any_cuda_call(lib):
    f = lib.fa_fwd_bwd_host
    vp, i = ctypes.c_void_p, ctypes.c_int
    f.argtypes = [vp] * 10 + [ctypes.c_size_t, i, i, i, i, i, ctypes.c_float, i, i, i, vp]
    f.restype = ctypes.c_int
    assert f(*([None] * 10), 0, 1, 2, 2, 128, 64, 0.125, 1, 0, 0, None) != 0
    lib.fa_last_error_message.restype = ctypes.c_char_p
    assert b"null" in lib.fa_last_error_message()


def test_release_and_debug_builds(lib):
    # the release library compiles the device index checks away; the FA_DEBUG build keeps them
    # (its kernels are exercised on the GPU by tests/test_gpu_debug_build.py)
    from exact_tiled_attention_07_gb300 import build as b

    lib.fa_debug_build.restype = ctypes.c_int
    assert lib.fa_debug_build() == 0
    dbg = ctypes.CDLL(b.build(debug=True))
    dbg.fa_debug_build.restype = ctypes.c_int
    assert dbg.fa_debug_build() == 1
