"""The persistent forward's work-item queues (a library-owned pool of counter slots).

A stream keeps the slot of its last launch; a stream without one takes a slot only once the
previous launch on it has finished; with every slot busy, or on a stream being captured into a
CUDA graph, a launch runs the static order instead.  Whichever
path runs, each item is computed the same way, so O and L equal a reference launch bit for bit.
"""

import pytest

from exact_tiled_attention_07_gb300.inputs import Workload, make_inputs
from helpers import to_device

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def fa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from exact_tiled_attention_07_gb300 import binding, build

    build.build()
    return binding


@pytest.fixture(scope="module")
def problem(fa):
    w = Workload("queue", 2, 8, 1536, 128, "bf16", True, "normal", 9700)
    x = make_inputs(w, with_do=False)
    dev = {key: to_device(val, w.dtype) for key, val in x.items()}
    o, lse = fa.attention_forward(dev["q"], dev["k"], dev["v"], causal=True, scale=w.scale)
    torch.cuda.synchronize()
    return w, dev, o, lse


def _launch(fa, w, dev):
    o = torch.empty_like(dev["q"])
    lse = torch.empty(dev["q"].shape[:3], dtype=torch.float32, device="cuda")
    fa.fa_fwd(dev["q"], dev["k"], dev["v"], o, lse, w.scale, True)
    return o, lse


def test_back_to_back_launches_on_one_stream_reuse_its_slot(fa, problem):
    w, dev, o_ref, l_ref = problem
    torch.cuda._sleep(50_000_000)  # holds the stream, so the launches below are all still pending
    outs = [_launch(fa, w, dev) for _ in range(40)]
    torch.cuda.synchronize()
    fa.fa_check_device_error()
    for o, lse in outs:
        assert torch.equal(o, o_ref) and torch.equal(lse, l_ref)


def test_more_streams_with_pending_launches_than_queue_slots(fa, problem):
    """40 streams, each holding a pending launch behind a sleep: more than the 32 slots, so the
    last streams find every slot busy and run the static order."""
    w, dev, o_ref, l_ref = problem
    streams = [torch.cuda.Stream() for _ in range(40)]
    outs = []
    for s in streams:
        with torch.cuda.stream(s):
            torch.cuda._sleep(20_000_000)
            outs.append(_launch(fa, w, dev))
    torch.cuda.synchronize()
    fa.fa_check_device_error()
    for o, lse in outs:
        assert torch.equal(o, o_ref) and torch.equal(lse, l_ref)


def test_launches_on_two_streams_at_once(fa, problem):
    w, dev, o_ref, l_ref = problem
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    outs = []
    for _ in range(6):
        for s in streams:
            with torch.cuda.stream(s):
                outs.append(_launch(fa, w, dev))
    torch.cuda.synchronize()
    fa.fa_check_device_error()
    for o, lse in outs:
        assert torch.equal(o, o_ref) and torch.equal(lse, l_ref)


def test_forward_captured_in_a_cuda_graph(fa, problem):
    w, dev, o_ref, l_ref = problem
    o = torch.empty_like(dev["q"])
    lse = torch.empty(dev["q"].shape[:3], dtype=torch.float32, device="cuda")
    fa.fa_fwd(dev["q"], dev["k"], dev["v"], o, lse, w.scale, True)  # warm up outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fa.fa_fwd(dev["q"], dev["k"], dev["v"], o, lse, w.scale, True)
    o.zero_()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    fa.fa_check_device_error()
    assert torch.equal(o, o_ref) and torch.equal(lse, l_ref)
