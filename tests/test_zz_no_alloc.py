"""fa_bwd_noalloc: the backward pass for callers that cannot allocate device memory.

Such callers (code inside a host application that owns every device allocation, or a
latency-bound loop that cannot afford cudaMalloc's implicit synchronisation) get their
scratch from a static device array in the library instead of a workspace argument.  The
test calls that entry point through the C ABI twice in a row (the second call finds the
first call's data in the shared array) and compares each result with fa_bwd given an
ordinary workspace, within the backward tolerance of the parity tests.  This file is
collected last so that a run stopping at the first failure has run everything else.
"""

import numpy as np
import pytest

from exact_tiled_attention_07_gb300.inputs import Workload, make_inputs
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


@pytest.mark.parametrize("w", [
    Workload("noalloc_bf16", 2, 2, 300, 128, "bf16", True, "normal", 8100),
    Workload("noalloc_fp16", 1, 3, 513, 64, "fp16", False, "normal", 8200),
])
def test_noalloc_matches_workspace_backward_twice(fa, w):
    x = {k: to_device(v, w.dtype) for k, v in make_inputs(w).items()}
    o, lse = fa.attention_forward(x["q"], x["k"], x["v"], causal=w.causal, scale=w.scale)
    ref = fa.attention_backward(x["q"], x["k"], x["v"], o, x["do"], lse, causal=w.causal, scale=w.scale)
    ref = [to_f64(t) for t in ref]
    for _ in range(2):
        got = [torch.full_like(x["q"], float("nan")) for _ in range(3)]
        fa.fa_bwd_noalloc(x["q"], x["k"], x["v"], o, x["do"], lse, got[0], got[1], got[2], w.scale, w.causal)
        fa.fa_check_device_error()
        for name, g, r in zip(("dq", "dk", "dv"), got, ref):
            g = to_f64(g)
            assert np.isfinite(g).all(), name
            assert rel_rms(g, r) <= TOL_GRAD_RELRMS, (name, rel_rms(g, r))


def test_noalloc_rejects_problems_beyond_the_static_scratch(fa):
    n = 4096
    assert fa.fa_bwd_workspace_size(8, 16, n, 128) > fa.NOALLOC_SCRATCH_BYTES
    t = torch.empty((8, 16, n, 128), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((8, 16, n), dtype=torch.float32, device="cuda")
    with pytest.raises(fa.FAError, match="scratch"):
        fa.fa_bwd_noalloc(t, t, t, t, t, lse, t, t, t, 0.125, True)
