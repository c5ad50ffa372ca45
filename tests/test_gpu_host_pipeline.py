"""fa_fwd_bwd_host: forward + backward over host buffers, chunked over key/value heads.

The chunked pipeline runs the same kernels on sub-batches of heads, so O, L, dK and dV must
equal the device-buffer path bit for bit (each is computed per head in an order that does not
depend on scheduling); dQ is a sum over key tiles reduced in scheduling order, so it is
compared with the fp64 oracle at the usual tolerance.  Chunks of 1, of a ragged 3, and the
automatic choice cover a last chunk smaller than the others.
"""

import numpy as np
import pytest

from oracle import gqa as G
from exact_tiled_attention_07_gb300.inputs import Workload, make_inputs, to_float64
from helpers import TOL_GRAD_RELRMS, TOL_L_MAXABS, TOL_O_MAXABS, TOL_O_RELRMS, max_abs, rel_rms, to_device, to_f64

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def fa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from exact_tiled_attention_07_gb300 import binding, build

    build.build()
    return binding


def _host(t):
    h = torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
    h.copy_(t)
    return h


def _run_host(fa, dev, w, chunk):
    q, k, v, do = (_host(dev[n]) for n in ("q", "k", "v", "do"))
    B, H, N, d = q.shape
    Hkv = k.shape[1]
    o, dq = torch.empty_like(q).pin_memory(), torch.empty_like(q).pin_memory()
    dk, dv = torch.empty_like(k).pin_memory(), torch.empty_like(k).pin_memory()
    lse = torch.empty((B, H, N), dtype=torch.float32).pin_memory()
    nbytes = fa.fa_fwd_bwd_host_workspace_size(B, H, Hkv, N, d, q.dtype, chunk)
    assert nbytes > 0
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    fa.fa_fwd_bwd_host(q, k, v, do, o, lse, dq, dk, dv, ws, w.scale, w.causal, chunk)
    torch.cuda.synchronize()
    fa.fa_check_device_error()
    return o, lse, dq, dk, dv


@pytest.mark.parametrize("chunk", [0, 1, 3])
@pytest.mark.parametrize("d,dtype,causal,b,h,hkv,n", [
    (64, "bf16", True, 2, 4, 2, 300),
    (128, "fp16", False, 1, 8, 8, 257),
    (128, "bf16", True, 3, 4, 4, 384),
    (64, "fp32", True, 1, 2, 2, 130),  # the CUDA-core kernels
    (64, "bf16", False, 4, 16, 16, 130),  # 64 key/value heads: eight automatic chunks of 8
])
def test_host_pipeline_matches_device_path(fa, chunk, d, dtype, causal, b, h, hkv, n):
    w = Workload("host", b, h, n, d, dtype, causal, "normal", 9500 + d + n, Hkv=hkv)
    x = make_inputs(w)
    dev = {key: to_device(val, w.dtype) for key, val in x.items()}
    o_d, l_d = fa.attention_forward(dev["q"], dev["k"], dev["v"], causal=w.causal, scale=w.scale)
    dq_d, dk_d, dv_d = fa.attention_backward(dev["q"], dev["k"], dev["v"], o_d, dev["do"], l_d, causal=w.causal,
                                             scale=w.scale)
    torch.cuda.synchronize()
    o, lse, dq, dk, dv = _run_host(fa, dev, w, chunk)
    for name, got, ref in (("O", o, o_d), ("L", lse, l_d), ("dK", dk, dk_d), ("dV", dv, dv_d)):
        assert torch.equal(got, ref.cpu()), name
    x64 = {key: to_float64(val, w.dtype) for key, val in x.items()}
    o_ref, l_ref = G.attn_fwd64_gqa(x64["q"], x64["k"], x64["v"], w.scale, w.causal)
    g_ref = G.attn_bwd64_gqa(x64["q"], x64["k"], x64["v"], x64["do"], w.scale, w.causal)[:3]
    assert max_abs(to_f64(o), o_ref) <= TOL_O_MAXABS and rel_rms(to_f64(o), o_ref) <= TOL_O_RELRMS
    assert max_abs(to_f64(lse), l_ref) <= TOL_L_MAXABS
    for name, got, ref in zip(("dq", "dk", "dv"), (dq, dk, dv), g_ref):
        assert rel_rms(to_f64(got), ref) <= TOL_GRAD_RELRMS, (name, rel_rms(to_f64(got), ref))


def test_host_pipeline_back_to_back_calls_reuse_the_streams(fa):
    """Two calls in a row on one workspace (the second must wait for the first's slots)."""
    w = Workload("host2", 2, 4, 256, 64, "bf16", True, "normal", 9600)
    x = make_inputs(w)
    dev = {key: to_device(val, w.dtype) for key, val in x.items()}
    first = _run_host(fa, dev, w, 1)
    q, k, v, do = (_host(dev[n]) for n in ("q", "k", "v", "do"))
    outs = [torch.empty_like(t).pin_memory() for t in first]
    ws = torch.empty(fa.fa_fwd_bwd_host_workspace_size(2, 4, 4, 256, 64, q.dtype, 1), dtype=torch.uint8,
                     device="cuda")
    for _ in range(2):
        fa.fa_fwd_bwd_host(q, k, v, do, outs[0], outs[1], outs[2], outs[3], outs[4], ws, w.scale, w.causal, 1)
    torch.cuda.synchronize()
    for name, a, b in zip(("O", "L", "dQ", "dK", "dV"), outs, first):
        if name == "dQ":
            assert rel_rms(to_f64(a), to_f64(b)) <= 1e-3
        else:
            assert torch.equal(a, b), name


def test_host_pipeline_rejects_a_small_workspace(fa):
    q = torch.zeros((1, 2, 128, 64), dtype=torch.bfloat16).pin_memory()
    lse = torch.zeros((1, 2, 128), dtype=torch.float32).pin_memory()
    need = fa.fa_fwd_bwd_host_workspace_size(1, 2, 2, 128, 64, q.dtype, 0)
    ws = torch.empty(need - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(fa.FAError, match="workspace"):
        fa.fa_fwd_bwd_host(q, q, q, q, q, lse, q, q, q, ws, 0.125, True, 0)
    with pytest.raises(ValueError, match="host"):
        fa.fa_fwd_bwd_host(q.cuda(), q, q, q, q, lse, q, q, q, ws, 0.125, True, 0)
