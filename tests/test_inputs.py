"""The seeded input generators (shared by the oracle's callers and the CUDA path's callers)."""

import numpy as np

from exact_tiled_attention_07_gb300.inputs import (
    DECODE_WORKLOADS,
    DecodeWorkload,
    f32_from_bf16_bits,
    make_decode_inputs,
    round_to_dtype,
)


def test_decode_workload_bytes():
    w = DECODE_WORKLOADS["decode_gqa_bf16"]
    cache = 2 * w.B * w.Hkv * w.Nk * w.d * 2
    assert cache == 1 << 30  # 8 x 8 heads x 32768 keys x 128 x 2 bytes, K and V
    rows = w.B * w.H * w.Nq
    assert w.bytes_moved() == cache + 2 * rows * w.d * 2 + 4 * rows


def test_decode_inputs_are_seeded_and_rounded():
    w = DecodeWorkload("small", 2, 4, 2, 3, 50, 64, "bf16", 7)
    a, b = make_decode_inputs(w), make_decode_inputs(w)
    assert a["q"].shape == (2, 4, 3, 64) and a["k"].shape == (2, 2, 50, 64) and a["v"].shape == (2, 2, 50, 64)
    for n in ("q", "k", "v"):
        assert np.array_equal(a[n], b[n])
        # stored values are bf16 already: rounding again changes nothing
        x = f32_from_bf16_bits(a[n])
        assert np.array_equal(round_to_dtype(x, "bf16"), a[n])
    assert not np.array_equal(a["k"], a["v"])
    w2 = DecodeWorkload("small", 2, 4, 2, 3, 50, 64, "bf16", 8)
    assert not np.array_equal(make_decode_inputs(w2)["q"], a["q"])


def test_bf16_rounding_matches_torch():
    """Round to nearest even, as torch's float32 -> bfloat16 conversion: random bit patterns
    (every exponent, infinities, NaNs, subnormals) and exact ties."""
    import torch

    from exact_tiled_attention_07_gb300.inputs import bf16_bits_from_f32

    rng = np.random.default_rng(11)
    bits = rng.integers(0, 2**32, size=1 << 20, dtype=np.uint64).astype(np.uint32)
    ties = (rng.integers(0, 2**16, size=4096, dtype=np.uint64).astype(np.uint32) << 16) | np.uint32(0x8000)
    x = np.concatenate([bits, ties]).view(np.float32)
    ours = bf16_bits_from_f32(x)
    ref = torch.from_numpy(x.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    nan = np.isnan(x)
    assert np.array_equal(ours[~nan], ref[~nan])
    assert np.all(ours[nan] == 0x7FC0)
