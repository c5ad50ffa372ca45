"""fa_bwd_noalloc: the backward pass for callers that cannot allocate device memory.

Such callers (code inside a host application that owns every device allocation, or a
latency-bound loop that cannot afford cudaMalloc's implicit synchronisation) get their
scratch from a static device array in the library instead of a workspace argument.  Every
call shares that array and finds the previous call's data in it, so the tests call the entry
point through the C ABI several times in a row, with different shapes, and check each result
three ways:

* dK and dV bit for bit against fa_bwd given an ordinary workspace (a key tile is one work
  item of one thread block, so both are deterministic);
* dQ against fa_bwd to the fp32 summation order (its partial sums reach the accumulator in
  whatever order the thread blocks finish): at most two units in the last place of the
  16-bit type, plus a part in a million of the largest element;
* dQ, dK, dV against the fp64 oracle at the backward tolerance of the parity tests, so a
  fault shared by both entry points fails too.

The size limit is tried on both sides: the largest problem whose workspace fits in the static
array runs and matches fa_bwd, and one 128-row block more is refused before anything runs.
This file is collected last so that a run stopping at the first failure has run everything
else.
"""

import numpy as np
import pytest

import oracle
from exact_tiled_attention_07_gb300.inputs import Workload, make_inputs, to_float64
from helpers import TOL_GRAD_RELRMS, rel_rms, to_device, to_f64

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def fa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from exact_tiled_attention_07_gb300 import binding, build

    build.build()
    return binding


def _ulp16(x, dtype):
    """Spacing of the 16-bit type at |x| (normal range; its smallest subnormal below it)."""
    mant, emin = (7, -126) if dtype == torch.bfloat16 else (10, -14)
    e = np.floor(np.log2(np.maximum(np.abs(x), 2.0 ** emin)))
    return 2.0 ** (e - mant)


def _case(w):
    x = make_inputs(w)
    dev = {k: to_device(v, w.dtype) for k, v in x.items()}
    return x, dev


def _noalloc_vs_workspace(fa, w, dev):
    """Run fa_bwd (own workspace) and fa_bwd_noalloc on the same inputs; check dK, dV bit for
    bit and dQ to the summation order; return the no-alloc results."""
    o, lse = fa.attention_forward(dev["q"], dev["k"], dev["v"], causal=w.causal, scale=w.scale)
    ref = fa.attention_backward(dev["q"], dev["k"], dev["v"], o, dev["do"], lse, causal=w.causal, scale=w.scale)
    got = [torch.full_like(dev["q"], float("nan")) for _ in range(3)]
    fa.fa_bwd_noalloc(dev["q"], dev["k"], dev["v"], o, dev["do"], lse, got[0], got[1], got[2], w.scale, w.causal)
    fa.fa_check_device_error()
    assert torch.equal(got[1], ref[1]), "dK differs from fa_bwd"
    assert torch.equal(got[2], ref[2]), "dV differs from fa_bwd"
    gq, rq = to_f64(got[0]), to_f64(ref[0])
    assert np.isfinite(gq).all()
    bound = 2 * _ulp16(rq, dev["q"].dtype) + 1e-6 * np.abs(rq).max()
    assert (np.abs(gq - rq) <= bound).all(), float(np.abs(gq - rq).max())
    return [to_f64(t) for t in got]


def _check_oracle(w, x, got):
    x64 = {k: to_float64(v, w.dtype) for k, v in x.items()}
    dq, dk, dv, _ = oracle.attn_bwd64(x64["q"], x64["k"], x64["v"], x64["do"], w.scale, w.causal)
    for name, g, r in zip(("dq", "dk", "dv"), got, (dq, dk, dv)):
        assert rel_rms(g, r) <= TOL_GRAD_RELRMS, (w.name, name, rel_rms(g, r))


def test_noalloc_calls_in_a_row_with_different_shapes(fa):
    """A larger causal bf16 d = 128 call, a smaller non-causal fp16 d = 64 call, a d = 256 call,
    then the first again: each finds the previous call's queue counters and accumulator rows in
    the array."""
    big = Workload("noalloc_bf16", 2, 2, 700, 128, "bf16", True, "normal", 8100)
    small = Workload("noalloc_fp16", 1, 3, 513, 64, "fp16", False, "normal", 8200)
    wide = Workload("noalloc_d256", 1, 2, 300, 256, "bf16", True, "normal", 8250)
    cases = {w.name: (w,) + _case(w) for w in (big, small, wide)}
    for name in ("noalloc_bf16", "noalloc_fp16", "noalloc_d256", "noalloc_bf16"):
        w, x, dev = cases[name]
        got = _noalloc_vs_workspace(fa, w, dev)
        _check_oracle(w, x, got)


def _largest_fitting_rows(fa, h, d):
    """N (a multiple of 128) of the largest B = 1, H = h problem whose workspace fits."""
    n = 128
    while fa.fa_bwd_workspace_size(1, h, n + 128, d) <= fa.NOALLOC_SCRATCH_BYTES:
        n += 128
    return n


def test_noalloc_at_and_just_beyond_the_size_limit(fa):
    h = 5
    n = _largest_fitting_rows(fa, h, 64)
    assert fa.fa_bwd_workspace_size(1, h, n, 64) <= fa.NOALLOC_SCRATCH_BYTES
    assert fa.fa_bwd_workspace_size(1, h, n + 128, 64) > fa.NOALLOC_SCRATCH_BYTES
    w = Workload("noalloc_limit", 1, h, n, 64, "bf16", True, "normal", 8300)
    x, dev = _case(w)
    got = _noalloc_vs_workspace(fa, w, dev)
    # dQ rows sampled over every head against the oracle (whole heads of this length are too
    # large for the fp64 definition on the host)
    rng = np.random.default_rng(8301)
    samples = np.stack([np.zeros(40, np.int64), rng.integers(0, h, 40), rng.integers(0, n, 40)], axis=1)
    samples = np.concatenate([samples, [[0, 0, 0], [0, h - 1, n - 1]]])
    ref = np.zeros((len(samples), 64))
    for hh in range(h):
        idx = np.nonzero(samples[:, 1] == hh)[0]
        if idx.size == 0:
            continue
        t = {nm: to_float64(x[nm][0, hh], w.dtype)[None, None] for nm in ("q", "k", "v", "do")}
        rows = np.stack([np.zeros_like(idx), np.zeros_like(idx), samples[idx, 2]], axis=1)
        ref[idx], _ = oracle.attn_bwd64_query_rows(t["q"], t["k"], t["v"], t["do"], w.scale, w.causal, rows)
    sampled = np.stack([got[0][0, hh, i] for _, hh, i in samples])
    assert rel_rms(sampled, ref) <= TOL_GRAD_RELRMS, rel_rms(sampled, ref)
    # one 128-row block more no longer fits: refused before anything runs
    t = torch.empty((1, h, n + 128, 64), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((1, h, n + 128), dtype=torch.float32, device="cuda")
    with pytest.raises(fa.FAError, match="scratch"):
        fa.fa_bwd_noalloc(t, t, t, t, t, lse, t, t, t, 0.125, True)


def test_noalloc_rejects_problems_far_beyond_the_static_scratch(fa):
    n = 4096
    assert fa.fa_bwd_workspace_size(8, 16, n, 128) > fa.NOALLOC_SCRATCH_BYTES
    t = torch.empty((8, 16, n, 128), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((8, 16, n), dtype=torch.float32, device="cuda")
    with pytest.raises(fa.FAError, match="scratch"):
        fa.fa_bwd_noalloc(t, t, t, t, t, lse, t, t, t, 0.125, True)
