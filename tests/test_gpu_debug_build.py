"""The FA_DEBUG build of the library: device-side index checks that record an error and never trap.

The debug library (``build.build(debug=True)``) is loaded in place of the release one for this
module and the release one is put back afterwards.  Small problems of every tensor-core path
(forward and backward at d = 64, 128 and 256, grouped-query heads, a sliding window, FP8 at
d = 64, 128 and 256) must run through it with no device error and match the fp64 oracle, so the checks
raise no false alarm; the self-test launches one check with an index out of range, which must
come back as a device error while the context stays usable.
"""

import numpy as np
import pytest

import oracle
from oracle import fp8 as F8
from oracle import gqa as G
from oracle import masks as M
from exact_tiled_attention_07_gb300.inputs import Workload, make_inputs, to_float64
from helpers import (TOL_GRAD_RELRMS, TOL_L_MAXABS, TOL_O_MAXABS, TOL_O_RELRMS, max_abs, rel_rms, to_device,
                     to_f64)

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def fa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from exact_tiled_attention_07_gb300 import binding, build

    release = build.build()
    debug = build.build(debug=True)
    binding.load_library(debug)
    try:
        assert binding.fa_debug_build()
        yield binding
    finally:
        binding.load_library(release)
        assert not binding.fa_debug_build()


def _check_fwd(w, x, o, lse, o_ref, l_ref):
    assert max_abs(to_f64(o), o_ref) <= TOL_O_MAXABS and rel_rms(to_f64(o), o_ref) <= TOL_O_RELRMS
    assert max_abs(to_f64(lse), l_ref) <= TOL_L_MAXABS


@pytest.mark.parametrize("d,dtype,causal", [(64, "fp16", False), (64, "bf16", True), (128, "bf16", True),
                                             (128, "fp16", False)])
def test_debug_build_forward_backward_parity(fa, d, dtype, causal):
    w = Workload("dbg", 2, 2, 300, d, dtype, causal, "normal", 7000 + d)
    x = make_inputs(w)
    dev = {k: to_device(v, w.dtype) for k, v in x.items()}
    o, lse = fa.attention_forward(dev["q"], dev["k"], dev["v"], causal=causal, scale=w.scale)
    dq, dk, dv = fa.attention_backward(dev["q"], dev["k"], dev["v"], o, dev["do"], lse, causal=causal, scale=w.scale)
    fa.fa_check_device_error()
    x64 = {k: to_float64(v, w.dtype) for k, v in x.items()}
    o_ref, l_ref = oracle.attn_fwd64(x64["q"], x64["k"], x64["v"], w.scale, causal)
    _check_fwd(w, x, o, lse, o_ref, l_ref)
    for g, r in zip((dq, dk, dv), oracle.attn_bwd64(x64["q"], x64["k"], x64["v"], x64["do"], w.scale, causal)[:3]):
        assert rel_rms(to_f64(g), r) <= TOL_GRAD_RELRMS


def test_debug_build_grouped_query_window_and_d256(fa):
    # grouped-query heads (4 query heads on 2 key/value heads), causal
    w = Workload("dbg_gqa", 1, 4, 260, 64, "bf16", True, "normal", 7100)
    x = make_inputs(w)
    q = to_device(x["q"], w.dtype)
    k, v = (to_device(np.ascontiguousarray(x[n][:, ::2]), w.dtype) for n in ("k", "v"))
    o, lse = fa.attention_forward(q, k, v, causal=True, scale=w.scale)
    fa.fa_check_device_error()
    o_ref, l_ref = G.attn_fwd64_gqa(to_float64(x["q"], "bf16"), to_float64(np.ascontiguousarray(x["k"][:, ::2]), "bf16"),
                                    to_float64(np.ascontiguousarray(x["v"][:, ::2]), "bf16"), w.scale, True)
    _check_fwd(w, x, o, lse, o_ref, l_ref)
    # a sliding window of 100 keys, causal
    w = Workload("dbg_win", 1, 2, 400, 128, "bf16", True, "normal", 7200)
    x = make_inputs(w, with_do=False)
    dev = {k_: to_device(v_, w.dtype) for k_, v_ in x.items()}
    o, lse = fa.attention_forward(dev["q"], dev["k"], dev["v"], causal=True, scale=w.scale, window=100)
    fa.fa_check_device_error()
    x64 = {k_: to_float64(v_, w.dtype) for k_, v_ in x.items()}
    o_ref, l_ref = M.attn_fwd64_masked(x64["q"], x64["k"], x64["v"], w.scale, M.visible_mask(w.N, causal=True,
                                                                                             window=100))
    _check_fwd(w, x, o, lse, o_ref, l_ref)
    # d = 256 forward and backward
    w = Workload("dbg_256", 1, 2, 300, 256, "bf16", True, "normal", 7300)
    x = make_inputs(w)
    dev = {k_: to_device(v_, w.dtype) for k_, v_ in x.items()}
    o, lse = fa.attention_forward(dev["q"], dev["k"], dev["v"], causal=True, scale=w.scale)
    dq, dk, dv = fa.attention_backward(dev["q"], dev["k"], dev["v"], o, dev["do"], lse, causal=True, scale=w.scale)
    fa.fa_check_device_error()
    x64 = {k_: to_float64(v_, w.dtype) for k_, v_ in x.items()}
    _check_fwd(w, x, o, lse, *oracle.attn_fwd64(x64["q"], x64["k"], x64["v"], w.scale, True))
    for g, r in zip((dq, dk, dv), oracle.attn_bwd64(x64["q"], x64["k"], x64["v"], x64["do"], w.scale, True)[:3]):
        assert rel_rms(to_f64(g), r) <= TOL_GRAD_RELRMS


@pytest.mark.parametrize("d,causal", [(64, False), (128, True), (256, False)])
def test_debug_build_fp8_forward(fa, d, causal):
    rng = np.random.default_rng(7400 + d)
    q, k, v = (rng.standard_normal((1, 2, 300, d)).astype(np.float32) for _ in range(3))
    host = [a for t in (q, k, v) for a in F8.quantize_blocks(t)]
    x8 = [fa.quantize_fp8(torch.from_numpy(t).cuda()) for t in (q, k, v)]
    o, lse = fa.attention_forward_fp8(*(c for c, _ in x8), *(s for _, s in x8), causal=causal)
    fa.fa_check_device_error()
    o_ref, l_ref = F8.attn_fwd64_fp8(*host, d ** -0.5, causal)
    assert rel_rms(to_f64(o), o_ref) <= 0.05


def test_debug_index_check_reports_and_the_context_survives(fa):
    fa.fa_selftest_debug_check(2, 3)
    fa.fa_check_device_error()  # in range: nothing recorded
    fa.fa_selftest_debug_check(5, 3)
    with pytest.raises(fa.FAError, match="index check failed"):
        fa.fa_check_device_error()
    fa.fa_check_device_error()  # the record was cleared by the read
    # the same context still computes
    w = Workload("dbg_after", 1, 1, 200, 64, "bf16", False, "normal", 7500)
    x = make_inputs(w, with_do=False)
    dev = {k_: to_device(v_, w.dtype) for k_, v_ in x.items()}
    o, lse = fa.attention_forward(dev["q"], dev["k"], dev["v"], scale=w.scale)
    fa.fa_check_device_error()
    x64 = {k_: to_float64(v_, w.dtype) for k_, v_ in x.items()}
    _check_fwd(w, x, o, lse, *oracle.attn_fwd64(x64["q"], x64["k"], x64["v"], w.scale, False))
