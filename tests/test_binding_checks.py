"""The Python binding refuses tensors the library cannot use, before any call into it: host
tensors (the C ABI takes device pointers), non-contiguous tensors, tensors on a GPU other than
the current one (the library launches on the current device), and a row statistic L of the
wrong type or size.  Runs on the CPU: every refusal happens before the library is loaded."""

from types import SimpleNamespace

import pytest

torch = pytest.importorskip("torch")

from exact_tiled_attention_07_gb300 import binding as fa  # noqa: E402


def _cpu(*shape, dtype=torch.bfloat16):
    return torch.zeros(shape, dtype=dtype)


B, H, N, D = 1, 2, 128, 64


@pytest.fixture
def host():
    t = _cpu(B, H, N, D)
    return {"t": t, "L": _cpu(B, H, N, dtype=torch.float32), "ws": _cpu(1 << 16, dtype=torch.uint8),
            "u8": _cpu(B, H, N, D, dtype=torch.uint8), "s": _cpu(B * H, dtype=torch.float32)}


def test_host_tensors_are_refused_by_every_device_entry_point(host):
    t, L, ws, u8, s = host["t"], host["L"], host["ws"], host["u8"], host["s"]
    calls = [
        lambda: fa.fa_fwd(t, t, t, t, L, 0.125, True),
        lambda: fa.fa_fwd_gqa(t, t, t, t, L, 0.125, True),
        lambda: fa.fa_bwd(t, t, t, t, t, L, t, t, t, ws, 0.125, True),
        lambda: fa.fa_bwd_gqa(t, t, t, t, t, L, t, t, t, ws, 0.125, True),
        lambda: fa.fa_bwd_noalloc(t, t, t, t, t, L, t, t, t, 0.125, True),
        lambda: fa.fa_bwd_preprocess(t, t, L, ws),
        lambda: fa.fa_bwd_main(t, t, t, t, t, t, ws, 0.125, True),
        lambda: fa.fa_bwd_dq_convert(ws, t, 0.125),
        lambda: fa.fa_fwd_masked(t, t, t, t, L, 0.125, True, window=64),
        lambda: fa.fa_bwd_masked(t, t, t, t, t, L, t, t, t, ws, 0.125, True, window=64),
        lambda: fa.fa_decode(t, t, t, t, L, 0.125),
        lambda: fa.fa_quantize_fp8(t, u8, s),
        lambda: fa.fa_fwd_fp8(u8, u8, u8, s, s, s, t, L, 0.125, True),
    ]
    for call in calls:
        with pytest.raises(ValueError, match="CUDA tensors"):
            call()


def test_host_pipeline_wants_its_workspace_on_the_device(host):
    t, L, ws = host["t"], host["L"], host["ws"]
    with pytest.raises(ValueError, match="device memory"):
        fa.fa_fwd_bwd_host(t, t, t, t, t, L, t, t, t, ws, 0.125, True)


def _fake(index, contiguous=True):
    return SimpleNamespace(is_cuda=True, is_contiguous=lambda: contiguous, device=SimpleNamespace(index=index))


def test_device_placement_rules(monkeypatch):
    monkeypatch.setattr(torch.cuda, "current_device", lambda: 0)
    fa._on_device(_fake(0), None, _fake(0))  # one GPU, the current one: accepted
    with pytest.raises(ValueError, match="contiguous"):
        fa._on_device(_fake(0), _fake(0, contiguous=False))
    with pytest.raises(ValueError, match="current device is cuda:0"):
        fa._on_device(_fake(1), _fake(1))
    with pytest.raises(ValueError, match="one GPU"):
        fa._on_device(_fake(0), _fake(1))


def test_row_statistic_type_and_size():
    fa._rows(_cpu(B, H, N, dtype=torch.float32), B * H * N)
    with pytest.raises(ValueError, match="fp32"):
        fa._rows(_cpu(B, H, N, dtype=torch.float16), B * H * N)
    with pytest.raises(ValueError, match="fp32"):
        fa._rows(_cpu(B, H, N - 1, dtype=torch.float32), B * H * N)
