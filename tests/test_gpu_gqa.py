"""Grouped-query and multi-query attention through the C ABI vs the fp64 oracle."""

import numpy as np
import pytest

from oracle import gqa as G
from exact_tiled_attention_07_gb300.inputs import Workload, make_inputs, to_float64
from helpers import (TOL_FP32, TOL_GRAD_RELRMS, TOL_L_MAXABS, TOL_O_MAXABS, TOL_O_RELRMS, max_abs, rel_rms,
                     to_device, to_f64)

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def fa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from exact_tiled_attention_07_gb300 import binding, build

    build.build()
    return binding


def _check(fa, w):
    x = make_inputs(w)
    dev = {k: to_device(v, w.dtype) for k, v in x.items()}
    o, lse = fa.attention_forward(dev["q"], dev["k"], dev["v"], causal=w.causal, scale=w.scale)
    dq, dk, dv = fa.attention_backward(dev["q"], dev["k"], dev["v"], o, dev["do"], lse, causal=w.causal,
                                       scale=w.scale)
    fa.fa_check_device_error()
    assert dk.shape == dev["k"].shape and dv.shape == dev["v"].shape
    x64 = {k: to_float64(v, w.dtype) for k, v in x.items()}
    o_ref, l_ref = G.attn_fwd64_gqa(x64["q"], x64["k"], x64["v"], w.scale, w.causal)
    g_ref = G.attn_bwd64_gqa(x64["q"], x64["k"], x64["v"], x64["do"], w.scale, w.causal)[:3]
    got = [to_f64(t) for t in (o, lse, dq, dk, dv)]
    if w.dtype == "fp32":
        for a, b in zip(got, (o_ref, l_ref) + tuple(g_ref)):
            assert max_abs(a, b) <= TOL_FP32
        return
    assert max_abs(got[0], o_ref) <= TOL_O_MAXABS and rel_rms(got[0], o_ref) <= TOL_O_RELRMS
    assert max_abs(got[1], l_ref) <= TOL_L_MAXABS
    for name, a, b in zip(("dq", "dk", "dv"), got[2:], g_ref):
        assert rel_rms(a, b) <= TOL_GRAD_RELRMS, (name, rel_rms(a, b))


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("h,hkv,n", [(4, 2, 300), (6, 1, 200), (8, 2, 129)])
def test_gqa_tensor_cores(fa, dtype, causal, d, h, hkv, n):
    _check(fa, Workload("gqa", 2, h, n, d, dtype, causal, "normal", 9000 + h * 10 + hkv, Hkv=hkv))


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("h,hkv,n", [(4, 2, 257), (4, 1, 130)])
def test_gqa_d256_forward_backward(fa, causal, h, hkv, n):
    # both halves of d of each key tile sum the gradients of every query head of the group
    _check(fa, Workload("gqa256b", 1, h, n, 256, "bf16", causal, "normal", 9150 + h + hkv + n, Hkv=hkv))


@pytest.mark.parametrize("causal", [False, True])
def test_gqa_forward_d256(fa, causal):
    w = Workload("gqa256", 1, 4, 257, 256, "bf16", causal, "normal", 9100, Hkv=2)
    x = make_inputs(w, with_do=False)
    dev = {k: to_device(v, w.dtype) for k, v in x.items()}
    o, lse = fa.attention_forward(dev["q"], dev["k"], dev["v"], causal=causal)
    x64 = {k: to_float64(v, w.dtype) for k, v in x.items()}
    o_ref, l_ref = G.attn_fwd64_gqa(x64["q"], x64["k"], x64["v"], w.scale, causal)
    assert max_abs(to_f64(o), o_ref) <= TOL_O_MAXABS and max_abs(to_f64(lse), l_ref) <= TOL_L_MAXABS


@pytest.mark.parametrize("causal", [False, True])
def test_gqa_fp32_and_cuda_core_path(fa, causal):
    _check(fa, Workload("gqa32", 1, 4, 70, 64, "fp32", causal, "normal", 9200, Hkv=2))
    _check(fa, Workload("gqa96", 1, 4, 90, 96, "bf16", causal, "normal", 9300, Hkv=1))


def test_gqa_rejects_heads_that_do_not_divide(fa):
    q = torch.empty((1, 4, 128, 64), dtype=torch.bfloat16, device="cuda")
    k = torch.empty((1, 3, 128, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ValueError):
        fa.attention_forward(q, k, k)
