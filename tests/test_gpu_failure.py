"""Failure detection without a GPU fault: a bounded wait that runs out is reported, and the
context stays usable afterwards."""

import pytest

import oracle
from exact_tiled_attention_07_gb300.inputs import Workload, make_inputs, to_float64
from helpers import TOL_L_MAXABS, TOL_O_MAXABS, max_abs, to_device, to_f64

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def fa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from exact_tiled_attention_07_gb300 import binding, build

    build.build()
    return binding


def test_expired_wait_is_reported_and_the_context_survives(fa):
    fa.fa_check_device_error()  # nothing pending
    fa.fa_selftest_bounded_wait(timeout_ms=20, arrive=False)
    with pytest.raises(fa.FAError) as e:
        fa.fa_check_device_error()
    assert e.value.status == 4 and "site 900" in str(e.value)
    fa.fa_check_device_error()  # the error word was cleared by the read
    # the control case records nothing
    fa.fa_selftest_bounded_wait(timeout_ms=20, arrive=True)
    fa.fa_check_device_error()
    # and the library still computes correct results on this context
    w = Workload("after", 1, 2, 200, 64, "bf16", True, "normal", 77)
    x = make_inputs(w, with_do=False)
    dev = {k: to_device(v, w.dtype) for k, v in x.items()}
    o, lse = fa.attention_forward(dev["q"], dev["k"], dev["v"], causal=True)
    fa.fa_check_device_error()
    x64 = {k: to_float64(v, w.dtype) for k, v in x.items()}
    o_ref, l_ref = oracle.attn_fwd64(x64["q"], x64["k"], x64["v"], w.scale, True)
    assert max_abs(to_f64(o), o_ref) <= TOL_O_MAXABS
    assert max_abs(to_f64(lse), l_ref) <= TOL_L_MAXABS
