"""The five workloads at full size, in the launch configuration bench.py times (and the
backward of the head-dimension-256 shape, which that workload does not time).

The GPU runs each whole problem; the oracle checks what it can compute exactly one by
one: every row of a few whole heads, a random sample of query rows (O, L, dQ) over all
heads, sampled key rows (dK, dV), plus properties that hold at any size and cost O(N d):
  * causal row 0 sees only key 0:  O_0 = V_0 and L_0 = tau q_0.k_0  (every head)
  * L_i >= tau q_i.k_j for any visible key j (log-sum-exp bounds each term): checked on
    the diagonal key j = i (causal) or key 0 (non-causal), every row of every head
  * every output finite.
"""

import numpy as np
import pytest

import oracle
from exact_tiled_attention_07_gb300.inputs import WORKLOADS, make_inputs, to_float64
from helpers import (TOL_GRAD_RELRMS, TOL_L_MAXABS, TOL_O_MAXABS, TOL_O_RELRMS, key_side_reference, max_abs,
                     oracle_pool_map, rel_rms, to_device, to_f64)

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def fa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from exact_tiled_attention_07_gb300 import binding, build

    build.build()
    return binding


def _run_full(fa, w):
    x = make_inputs(w, with_do=not w.fwd_only)
    dev = {k: to_device(v, w.dtype) for k, v in x.items()}
    o, lse = fa.attention_forward(dev["q"], dev["k"], dev["v"], causal=w.causal, scale=w.scale)
    out = {"o": o, "lse": lse}
    if not w.fwd_only:
        dq, dk, dv = fa.attention_backward(dev["q"], dev["k"], dev["v"], o, dev["do"], lse, causal=w.causal,
                                           scale=w.scale)
        out.update(dq=dq, dk=dk, dv=dv)
    fa.fa_check_device_error()
    for name, t in out.items():
        assert bool(torch.isfinite(t).all()), name
    host = {k: v.cpu() for k, v in out.items()}
    del dev, out
    torch.cuda.empty_cache()
    return x, host


def _sample(w, count, seed):
    rng = np.random.default_rng(seed)
    flat = rng.choice(w.B * w.H * w.N, size=count, replace=False)
    s = np.stack([flat // (w.H * w.N), (flat // w.N) % w.H, flat % w.N], axis=1)
    edge = [(0, 0, 0), (0, 0, 1), (0, 0, 127), (0, 0, 128), (0, 0, w.N - 1), (w.B - 1, w.H - 1, w.N - 1)]
    return np.concatenate([s, np.array(edge)], axis=0)


def _take(t, samples):
    """Rows (b, h, i) of a host tensor [B, H, N, ...] as float64 numpy."""
    idx = [torch.as_tensor(samples[:, j], dtype=torch.long) for j in range(3)]
    return to_f64(t[idx[0], idx[1], idx[2]])


def _head64(w, x, name, b, h):
    return to_float64(x[name][b, h], w.dtype)


def _check_properties(w, x, host):
    lse_all = host["lse"]
    for b in range(w.B):
        for h in range(w.H):
            q, k = _head64(w, x, "q", b, h), _head64(w, x, "k", b, h)
            lse = to_f64(lse_all[b, h])
            if w.causal:
                diag = w.scale * (q * k).sum(-1)  # tau q_i.k_i, a visible term of row i
                assert (lse >= diag - 1e-3).all(), (b, h)
                assert abs(lse[0] - diag[0]) <= TOL_L_MAXABS, (b, h)
                v0 = to_float64(x["v"][b, h, 0], w.dtype)
                assert max_abs(to_f64(host["o"][b, h, 0]), v0) <= TOL_O_MAXABS, (b, h)
            else:
                first = w.scale * (q @ k[0])
                assert (lse >= first - 1e-3).all(), (b, h)


def _check_sampled_rows(w, x, host, samples, with_bwd):
    """O, L (and dQ) of sampled query rows, one head's inputs converted at a time."""
    got_o = _take(host["o"], samples)
    got_l = _take(host["lse"], samples)
    o_ref = np.zeros_like(got_o)
    l_ref = np.zeros_like(got_l)
    dq_ref = np.zeros_like(got_o)
    heads = sorted({(int(b), int(h)) for b, h, _ in samples})
    for b, h in heads:
        idx = np.nonzero((samples[:, 0] == b) & (samples[:, 1] == h))[0]
        rows = np.stack([np.zeros_like(idx), np.zeros_like(idx), samples[idx, 2]], axis=1)
        names = ("q", "k", "v", "do") if with_bwd else ("q", "k", "v")
        t = {nm: _head64(w, x, nm, b, h)[None, None] for nm in names}
        o_ref[idx], l_ref[idx] = oracle.attn_fwd64_rows(t["q"], t["k"], t["v"], w.scale, w.causal, rows)
        if with_bwd:
            dq_ref[idx], _ = oracle.attn_bwd64_query_rows(t["q"], t["k"], t["v"], t["do"], w.scale, w.causal, rows)
    assert max_abs(got_o, o_ref) <= TOL_O_MAXABS, max_abs(got_o, o_ref)
    assert rel_rms(got_o, o_ref) <= TOL_O_RELRMS, rel_rms(got_o, o_ref)
    assert max_abs(got_l, l_ref) <= TOL_L_MAXABS, max_abs(got_l, l_ref)
    if with_bwd:
        got = _take(host["dq"], samples)
        assert rel_rms(got, dq_ref) <= TOL_GRAD_RELRMS, rel_rms(got, dq_ref)


def _check_whole_heads(w, x, host, heads):
    for b, h in heads:
        q, k, v = (_head64(w, x, nm, b, h)[None, None] for nm in ("q", "k", "v"))
        o_ref, l_ref = oracle.attn_fwd64(q, k, v, w.scale, w.causal)
        go, gl = to_f64(host["o"][b, h]), to_f64(host["lse"][b, h])
        assert max_abs(go, o_ref[0, 0]) <= TOL_O_MAXABS and rel_rms(go, o_ref[0, 0]) <= TOL_O_RELRMS
        assert max_abs(gl, l_ref[0, 0]) <= TOL_L_MAXABS
        if not w.fwd_only:
            do = _head64(w, x, "do", b, h)[None, None]
            dq, dk, dv, _ = oracle.attn_bwd64(q, k, v, do, w.scale, w.causal)
            for name, ref in (("dq", dq), ("dk", dk), ("dv", dv)):
                got = to_f64(host[name][b, h])
                assert rel_rms(got, ref[0, 0]) <= TOL_GRAD_RELRMS, (name, b, h, rel_rms(got, ref[0, 0]))


def test_gpt2_medium_fp16(fa):
    w = WORKLOADS["gpt2m_fp16"]
    x, host = _run_full(fa, w)
    _check_properties(w, x, host)
    _check_whole_heads(w, x, host, [(0, 0), (31, 7), (63, 15)])
    _check_sampled_rows(w, x, host, _sample(w, 256, 21), with_bwd=True)


def test_causal_lm_bf16(fa):
    w = WORKLOADS["causal_lm_bf16"]
    x, host = _run_full(fa, w)
    _check_properties(w, x, host)
    _check_whole_heads(w, x, host, [(0, 0), (7, 15)])
    _check_sampled_rows(w, x, host, _sample(w, 256, 31), with_bwd=True)


def test_causal_lm_bf16_noncausal_variant(fa):
    # the same shape without the mask: the headline throughput case of the bench
    w = WORKLOADS["causal_lm_bf16"].with_shape(causal=False, seed=32)
    x, host = _run_full(fa, w)
    _check_properties(w, x, host)
    _check_whole_heads(w, x, host, [(3, 5)])
    _check_sampled_rows(w, x, host, _sample(w, 128, 33), with_bwd=True)


def test_long_sequence_causal_bf16(fa):
    w = WORKLOADS["long_causal_bf16"]
    x, host = _run_full(fa, w)
    _check_properties(w, x, host)
    _check_sampled_rows(w, x, host, _sample(w, 256, 41), with_bwd=True)
    # key-side gradients: 32 keys in each of the 8 heads (256 in all), random ones plus keys at
    # tile edges (0, 127, 128, 129, N - 129, N - 128, N - 1); each head's exact values need
    # every row's L and D of that head, so the heads run in a pool of worker processes
    rng = np.random.default_rng(42)
    edges = np.array([0, 127, 128, 129, w.N - 129, w.N - 128, w.N - 1])
    jobs, keys_of = [], {}
    for h in range(w.H):
        rnd = rng.choice(np.setdiff1d(np.arange(w.N), edges), 32 - edges.size, replace=False)
        keys = np.sort(np.concatenate([rnd, edges]))
        keys_of[h] = keys
        q, k, v, do = (_head64(w, x, nm, 0, h)[None, None] for nm in ("q", "k", "v", "do"))
        jobs.append((q, k, v, do, w.scale, w.causal, keys))
    refs = oracle_pool_map(key_side_reference, jobs)
    got_k, got_v, ref_k, ref_v = [], [], [], []
    for h, (dk_ref, dv_ref, l_ref) in enumerate(refs):
        kt = torch.as_tensor(keys_of[h], dtype=torch.long)
        got_k.append(to_f64(host["dk"][0, h][kt]))
        got_v.append(to_f64(host["dv"][0, h][kt]))
        ref_k.append(dk_ref)
        ref_v.append(dv_ref)
        assert max_abs(to_f64(host["lse"][0, h]), l_ref) <= TOL_L_MAXABS, h  # every row's L of the head
    assert sum(len(k_) for k_ in keys_of.values()) >= 256
    assert rel_rms(np.concatenate(got_k), np.concatenate(ref_k)) <= TOL_GRAD_RELRMS
    assert rel_rms(np.concatenate(got_v), np.concatenate(ref_v)) <= TOL_GRAD_RELRMS
    for h in range(w.H):  # and head by head
        assert rel_rms(got_k[h], ref_k[h]) <= TOL_GRAD_RELRMS, h
        assert rel_rms(got_v[h], ref_v[h]) <= TOL_GRAD_RELRMS, h


def test_head_dim_256_forward_bf16(fa):
    w = WORKLOADS["hd256_bf16"]
    x, host = _run_full(fa, w)
    _check_properties(w, x, host)
    _check_sampled_rows(w, x, host, _sample(w, 512, 51), with_bwd=False)


def test_head_dim_256_backward_full_size_sampled(fa):
    # the head-dimension-256 shape (B 4, H 16, N 16384) with its backward on the tensor cores:
    # query-side rows (O, L, dQ) sampled over all heads, key-side rows (dK, dV) of 16 keys in each
    # of four heads (random keys plus tile edges), each head's exact statistics in a worker pool
    w = WORKLOADS["hd256_bf16"].with_shape(fwd_only=False, seed=52)
    x, host = _run_full(fa, w)
    _check_sampled_rows(w, x, host, _sample(w, 96, 53), with_bwd=True)
    rng = np.random.default_rng(54)
    edges = np.array([0, 31, 32, 127, 128, w.N - 129, w.N - 1])
    heads = [(0, 0), (1, 7), (2, 11), (3, 15)]
    jobs, keys_of = [], {}
    for b, h in heads:
        rnd = rng.choice(np.setdiff1d(np.arange(w.N), edges), 16 - edges.size, replace=False)
        keys = np.sort(np.concatenate([rnd, edges]))
        keys_of[(b, h)] = keys
        q, k, v, do = (_head64(w, x, nm, b, h)[None, None] for nm in ("q", "k", "v", "do"))
        jobs.append((q, k, v, do, w.scale, w.causal, keys))
    refs = oracle_pool_map(key_side_reference, jobs)
    for (b, h), (dk_ref, dv_ref, l_ref) in zip(heads, refs):
        kt = torch.as_tensor(keys_of[(b, h)], dtype=torch.long)
        assert rel_rms(to_f64(host["dk"][b, h][kt]), dk_ref) <= TOL_GRAD_RELRMS, (b, h)
        assert rel_rms(to_f64(host["dv"][b, h][kt]), dv_ref) <= TOL_GRAD_RELRMS, (b, h)
        assert max_abs(to_f64(host["lse"][b, h]), l_ref) <= TOL_L_MAXABS, (b, h)
