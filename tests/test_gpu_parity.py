"""CUDA path vs the fp64 oracle, element by element, at sizes the oracle finishes in seconds.

All calls go through the C ABI (``exact_tiled_attention_07_gb300.binding``).  Shapes span
several 128-row tiles plus ragged tails, both masks, all three dtypes and the head
dimensions of the tensor-core kernels and of the CUDA-core path.
"""

import math

import numpy as np
import pytest

import oracle
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


def _run(fa, w, with_bwd=True):
    x = make_inputs(w, with_do=with_bwd)
    dev = {k: to_device(v, w.dtype) for k, v in x.items()}
    o, lse = fa.attention_forward(dev["q"], dev["k"], dev["v"], causal=w.causal, scale=w.scale)
    out = {"o": o, "lse": lse}
    if with_bwd:
        dq, dk, dv = fa.attention_backward(dev["q"], dev["k"], dev["v"], o, dev["do"], lse, causal=w.causal,
                                           scale=w.scale)
        out.update(dq=dq, dk=dk, dv=dv)
    fa.fa_check_device_error()
    x64 = {k: to_float64(v, w.dtype) for k, v in x.items()}
    return x64, {k: to_f64(v) for k, v in out.items()}


def _check_fwd(w, x64, got, fp32=False):
    o_ref, l_ref = oracle.attn_fwd64(x64["q"], x64["k"], x64["v"], w.scale, w.causal)
    assert np.isfinite(got["o"]).all() and np.isfinite(got["lse"]).all()
    if fp32:
        assert max_abs(got["o"], o_ref) <= TOL_FP32
        assert max_abs(got["lse"], l_ref) <= TOL_FP32
    else:
        assert max_abs(got["o"], o_ref) <= TOL_O_MAXABS, max_abs(got["o"], o_ref)
        assert rel_rms(got["o"], o_ref) <= TOL_O_RELRMS, rel_rms(got["o"], o_ref)
        assert max_abs(got["lse"], l_ref) <= TOL_L_MAXABS, max_abs(got["lse"], l_ref)


def _check_bwd(w, x64, got, fp32=False):
    dq, dk, dv, _ = oracle.attn_bwd64(x64["q"], x64["k"], x64["v"], x64["do"], w.scale, w.causal)
    for name, ref in (("dq", dq), ("dk", dk), ("dv", dv)):
        g = got[name]
        assert np.isfinite(g).all(), name
        if fp32:
            assert max_abs(g, ref) <= TOL_FP32, (name, max_abs(g, ref))
        else:
            assert rel_rms(g, ref) <= TOL_GRAD_RELRMS, (name, rel_rms(g, ref))


def test_tiny_fp32_config(fa):
    # 1 x 1 x 128 x 64, fp32, non-causal, seed 0: forward and backward within 1e-5
    w = Workload("tiny_fp32", 1, 1, 128, 64, "fp32", False, "normal", 0)
    x64, got = _run(fa, w)
    _check_fwd(w, x64, got, fp32=True)
    _check_bwd(w, x64, got, fp32=True)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("n,d", [(1, 64), (33, 64), (200, 128), (100, 32), (77, 256)])
def test_fp32_path(fa, n, d, causal):
    w = Workload("fp32", 1, 2, n, d, "fp32", causal, "normal", 11 + n)
    x64, got = _run(fa, w)
    _check_fwd(w, x64, got, fp32=True)
    _check_bwd(w, x64, got, fp32=True)


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("n", [1, 17, 128, 129, 255, 384, 700])
def test_tensor_core_fwd_bwd(fa, dtype, causal, d, n):
    w = Workload("tc", 2, 2, n, d, dtype, causal, "normal", 1000 + n + d)
    assert fa.fa_uses_tensor_cores("fwd", 0 if dtype == "bf16" else 1, d)
    x64, got = _run(fa, w)
    _check_fwd(w, x64, got)
    _check_bwd(w, x64, got)


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("n", [1, 130, 300, 512])
def test_tensor_core_fwd_d256(fa, dtype, causal, n):
    w = Workload("tc256", 1, 2, n, 256, dtype, causal, "normal", 2000 + n)
    x64, got = _run(fa, w, with_bwd=False)
    _check_fwd(w, x64, got)


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("n", [1, 31, 130, 300, 515])
def test_tensor_core_bwd_d256(fa, dtype, causal, n):
    # d = 256 backward on the tensor cores: each key tile's dK, dV in two halves of d (two work
    # items recomputing S and dP over all of d), 32 queries a step; ragged N and one-row problems
    w = Workload("tcb256", 2, 2, n, 256, dtype, causal, "normal", 2100 + n + causal)
    assert fa.fa_uses_tensor_cores("bwd", torch.bfloat16 if dtype == "bf16" else torch.float16, 256)
    x64, got = _run(fa, w)
    assert fa.fa_last_error_message() == ""  # no CUDA-core notice
    # the forward's element-wise bound is checked by the forward tests; here the rows of a few
    # keys (n = 31, causal) reach |O| > 2, where a bf16 output's own rounding is up to 2^-7
    o_ref, l_ref = oracle.attn_fwd64(x64["q"], x64["k"], x64["v"], w.scale, w.causal)
    assert rel_rms(got["o"], o_ref) <= TOL_O_RELRMS and max_abs(got["lse"], l_ref) <= TOL_L_MAXABS
    _check_bwd(w, x64, got)


@pytest.mark.parametrize("d", [32, 96, 200])
def test_cuda_core_path_16bit(fa, d):
    # head dims without a tensor-core kernel use the CUDA-core kernels; the binding warns about
    # it before the call
    w = Workload("simt16", 1, 2, 150, d, "bf16", True, "normal", 3000 + d)
    with pytest.warns(UserWarning, match="CUDA-core"):
        x64, got = _run(fa, w)
    _check_fwd(w, x64, got)
    _check_bwd(w, x64, got)


@pytest.mark.parametrize("d,pass_", [(96, "forward"), (200, "backward"), (32, "backward")])
def test_cuda_core_path_is_reported_by_the_c_abi(fa, d, pass_):
    # a 16-bit call that runs on the CUDA-core kernels succeeds and leaves a notice naming the
    # path; a tensor-core call leaves none
    w = Workload("notice", 1, 1, 130, d, "fp16", False, "normal", 3100 + d)
    x = {k: to_device(v, w.dtype) for k, v in make_inputs(w).items()}
    o = torch.empty_like(x["q"])
    lse = torch.empty((1, 1, 130), dtype=torch.float32, device="cuda")
    fa.fa_fwd(x["q"], x["k"], x["v"], o, lse, w.scale, False)
    if pass_ == "forward":
        msg = fa.fa_last_error_message()
        assert msg.startswith("notice:") and "forward" in msg and f"d={d}" in msg, msg
        return
    fwd_msg = fa.fa_last_error_message()
    assert (fwd_msg == "") == fa.fa_uses_tensor_cores("fwd", torch.float16, d), fwd_msg
    dq, dk, dv = (torch.empty_like(x["q"]) for _ in range(3))
    ws = torch.empty(fa.fa_bwd_workspace_size(1, 1, 130, d), dtype=torch.uint8, device="cuda")
    fa.fa_bwd(x["q"], x["k"], x["v"], o, x["do"], lse, dq, dk, dv, ws, w.scale, False)
    msg = fa.fa_last_error_message()
    assert msg.startswith("notice:") and "backward" in msg and f"d={d}" in msg, msg
    fa.fa_check_device_error()
    # a tensor-core call clears it
    w2 = Workload("notice_tc", 1, 1, 130, 64, "fp16", False, "normal", 3200)
    x2 = {k: to_device(v, w2.dtype) for k, v in make_inputs(w2, with_do=False).items()}
    fa.fa_fwd(x2["q"], x2["k"], x2["v"], torch.empty_like(x2["q"]), lse, w2.scale, False)
    assert fa.fa_last_error_message() == ""


def test_large_score_offsets_stress_rescaling(fa):
    # per-key offsets of the long-sequence workload at a small size: many max updates
    w = Workload("offsets", 1, 2, 640, 64, "bf16", True, "normal_key_offset", 4000)
    x64, got = _run(fa, w)
    _check_fwd(w, x64, got)
    _check_bwd(w, x64, got)


def test_forward_is_deterministic(fa):
    w = Workload("det", 2, 2, 384, 128, "bf16", True, "normal", 5000)
    x = {k: to_device(v, w.dtype) for k, v in make_inputs(w, with_do=False).items()}
    o1, l1 = fa.attention_forward(x["q"], x["k"], x["v"], causal=True)
    o2, l2 = fa.attention_forward(x["q"], x["k"], x["v"], causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_outputs_leave_guard_bands_untouched(fa):
    # outputs written into the middle of larger buffers: the guard bands must keep their pattern
    w = Workload("guard", 1, 2, 200, 64, "bf16", True, "normal", 6000)
    x = {k: to_device(v, w.dtype) for k, v in make_inputs(w).items()}
    numel = x["q"].numel()
    pad = 4096
    bufs = {}
    for name in ("o", "dq", "dk", "dv"):
        big = torch.full((numel + 2 * pad,), 7.0, dtype=torch.bfloat16, device="cuda")
        bufs[name] = (big, big[pad:pad + numel].view_as(x["q"]))
    lbig = torch.full((x["q"].shape[0] * 2 * 200 + 2 * pad,), 7.0, dtype=torch.float32, device="cuda")
    lse = lbig[pad:pad + 2 * 200].view(1, 2, 200)
    fa.fa_fwd(x["q"], x["k"], x["v"], bufs["o"][1], lse, w.scale, True)
    ws = torch.empty(fa.fa_bwd_workspace_size(1, 2, 200, 64), dtype=torch.uint8, device="cuda")
    fa.fa_bwd(x["q"], x["k"], x["v"], bufs["o"][1], x["do"], lse, bufs["dq"][1], bufs["dk"][1], bufs["dv"][1], ws,
              w.scale, True)
    fa.fa_check_device_error()
    for name, (big, _) in bufs.items():
        assert bool((big[:pad] == 7.0).all()) and bool((big[pad + numel:] == 7.0).all()), name
    assert bool((lbig[:pad] == 7.0).all()) and bool((lbig[pad + 400:] == 7.0).all())


def test_causal_tile_count(fa):
    # 128 x 128 score tiles visited by the causal forward: T (T + 1) / 2 per head
    n = 4096
    w = Workload("tiles", 1, 2, n, 64, "bf16", True, "normal", 7000)
    x = {k: to_device(v, w.dtype) for k, v in make_inputs(w, with_do=False).items()}
    fa.fa_tile_counter(reset=True)
    fa.attention_forward(x["q"], x["k"], x["v"], causal=True)
    t = n // 128
    assert fa.fa_tile_counter(reset=True) == 2 * oracle.causal_tiles_visited(n, 128, 128) == 2 * t * (t + 1) // 2
    fa.attention_forward(x["q"], x["k"], x["v"], causal=False)
    assert fa.fa_tile_counter(reset=True) == 2 * t * t


def test_empty_problem_is_a_no_op(fa):
    q = torch.empty((0, 4, 128, 64), dtype=torch.bfloat16, device="cuda")
    o, lse = fa.attention_forward(q, q, q)
    assert o.numel() == 0 and lse.numel() == 0
