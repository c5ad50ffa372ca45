"""Seeded synthetic inputs shared by the CUDA path's callers and the oracle.

This module holds no attention arithmetic: it draws random numbers, rounds
them to the storage dtype (round-to-nearest-even) and names the workloads.
Both the oracle (through the tests and the CPU baseline) and the CUDA path
consume exactly the arrays it returns.

Workloads (shapes B, H, N, d; all scale τ = 1/√d):

* ``tiny_fp32``       1, 1, 128, 64,   fp32, non-causal, Q, K, V, dO ~ N(0,1), seed 0
* ``gpt2m_fp16``      64, 16, 1024, 64, fp16, non-causal, every element N(0,1)/√d
  (GPT-2-medium attention, the workload of "FlashAttention and GPU memory" §01/§09)
* ``causal_lm_bf16``  8, 16, 4096, 128, bf16, causal, N(0,1)
* ``long_causal_bf16`` 1, 8, 65536, 64, bf16, causal, N(0,1) with a per-key score
  offset c_j ~ N(0, 4) realised through the inputs: Q[..., 0] = 1 and
  K[..., j, 0] = c_j·√d, so τ·q_i·k_j gains exactly c_j (stresses rescaling)
* ``hd256_bf16``      4, 16, 16384, 256, bf16, non-causal, forward only, N(0,1)

Decode workloads (``DECODE_WORKLOADS``: new query rows Q [B, H, Nq, d] against a key/value
cache K, V [B, Hkv, Nk, d]):

* ``decode_gqa_bf16`` 8, 32 query heads on 8 key/value heads, 1 new row, 32768 cached
  keys, d = 128, bf16, N(0,1), seed 600 (a 1.07 GB cache, larger than L2)

Random numbers come from numpy's PCG64 generator, drawn in float32 in the
order Q, K, V, dO, then the key offsets.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

__all__ = ["Workload", "WORKLOADS", "DecodeWorkload", "DECODE_WORKLOADS", "make_decode_inputs", "make_inputs", "round_to_dtype", "to_float64",
           "bf16_bits_from_f32", "f32_from_bf16_bits", "attention_flops"]

DTYPES = ("fp32", "fp16", "bf16")


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int
    d: int
    dtype: str
    causal: bool
    dist: str = "normal"  # "normal" | "normal_over_sqrt_d" | "normal_key_offset"
    seed: int = 0
    fwd_only: bool = False
    extra: dict = field(default_factory=dict)
    Hkv: int = 0  # key/value heads (grouped-query attention); 0 means H

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def kv_heads(self) -> int:
        return self.Hkv or self.H

    def with_shape(self, **kw) -> "Workload":
        fields = dict(name=self.name, B=self.B, H=self.H, N=self.N, d=self.d, dtype=self.dtype,
                      causal=self.causal, dist=self.dist, seed=self.seed, fwd_only=self.fwd_only, Hkv=self.Hkv)
        fields.update(kw)
        return Workload(**fields)


WORKLOADS = {
    "tiny_fp32": Workload("tiny_fp32", 1, 1, 128, 64, "fp32", False, "normal", 0),
    "gpt2m_fp16": Workload("gpt2m_fp16", 64, 16, 1024, 64, "fp16", False, "normal_over_sqrt_d", 1),
    "causal_lm_bf16": Workload("causal_lm_bf16", 8, 16, 4096, 128, "bf16", True, "normal", 2),
    "long_causal_bf16": Workload("long_causal_bf16", 1, 8, 65536, 64, "bf16", True, "normal_key_offset", 3),
    "hd256_bf16": Workload("hd256_bf16", 4, 16, 16384, 256, "bf16", False, "normal", 4, fwd_only=True),
}


def bf16_bits_from_f32(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (nearest, ties to even); returns the uint16 bit patterns."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    flat_u = x.reshape(-1).view(np.uint32)
    flat_x = x.reshape(-1)
    r = np.empty(flat_u.shape, dtype=np.uint16)
    step = 1 << 22  # slices small enough that the temporaries stay in cache
    for i in range(0, flat_u.size, step):
        u = flat_u[i:i + step]
        t = u >> np.uint32(16)  # (u + 0x7FFF + lsb) >> 16
        t &= np.uint32(1)
        t += np.uint32(0x7FFF)
        t += u
        t >>= np.uint32(16)
        ri = r[i:i + step]
        ri[...] = t
        nan = np.isnan(flat_x[i:i + step])
        if nan.any():
            ri[nan] = np.uint16(0x7FC0)
    return r.reshape(x.shape)


def f32_from_bf16_bits(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def round_to_dtype(x: np.ndarray, dtype: str) -> np.ndarray:
    """Storage array for ``dtype``: float32, float16, or uint16 bf16 bit patterns."""
    if dtype == "fp32":
        return np.ascontiguousarray(x, dtype=np.float32)
    if dtype == "fp16":
        return np.ascontiguousarray(x, dtype=np.float32).astype(np.float16)
    if dtype == "bf16":
        return bf16_bits_from_f32(np.asarray(x, dtype=np.float32))
    raise ValueError(f"unknown dtype {dtype!r}")


def to_float64(stored: np.ndarray, dtype: str) -> np.ndarray:
    """Exact float64 values of a storage array produced by ``round_to_dtype``."""
    if dtype == "bf16":
        return f32_from_bf16_bits(stored).astype(np.float64)
    return np.asarray(stored).astype(np.float64)


def make_inputs(w: Workload, with_do: bool = True) -> dict:
    """Draw Q, K, V (and dO) for workload ``w``; values already rounded to ``w.dtype``.

    Returns a dict of storage arrays under keys q, k, v, do: Q and dO [B, H, N, d], K and V
    [B, H_kv, N, d] (H_kv = H unless the workload shares key/value heads).
    """
    rng = np.random.Generator(np.random.PCG64(w.seed))
    shape = (w.B, w.H, w.N, w.d)
    kv_shape = (w.B, w.kv_heads, w.N, w.d)
    names = ["q", "k", "v"] + (["do"] if with_do else [])
    raw = {}
    for nm in names:
        raw[nm] = rng.standard_normal(size=kv_shape if nm in ("k", "v") else shape, dtype=np.float32)
    if w.dist == "normal_over_sqrt_d":
        f = np.float32(1.0 / math.sqrt(w.d))
        for nm in names:
            raw[nm] *= f
    elif w.dist == "normal_key_offset":
        # per-key additive score offset c_j ~ N(0, σ² = 4), carried by coordinate 0
        c = rng.standard_normal(size=(w.B, w.kv_heads, w.N), dtype=np.float32) * np.float32(2.0)
        raw["q"][..., 0] = 1.0
        raw["k"][..., 0] = c * np.float32(math.sqrt(w.d))
    elif w.dist != "normal":
        raise ValueError(f"unknown distribution {w.dist!r}")
    return {nm: round_to_dtype(a, w.dtype) for nm, a in raw.items()}


@dataclass(frozen=True)
class DecodeWorkload:
    name: str
    B: int
    H: int
    Hkv: int
    Nq: int
    Nk: int
    d: int
    dtype: str = "bf16"
    seed: int = 0

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    def bytes_moved(self) -> int:
        """Compulsory HBM bytes of one decode step: read Q, K, V; write O (dtype) and L (fp32)."""
        e = 4 if self.dtype == "fp32" else 2
        rows = self.B * self.H * self.Nq
        return e * (2 * self.B * self.Hkv * self.Nk * self.d + 2 * rows * self.d) + 4 * rows


DECODE_WORKLOADS = {
    "decode_gqa_bf16": DecodeWorkload("decode_gqa_bf16", 8, 32, 8, 1, 32768, 128, "bf16", 600),
}


def make_decode_inputs(w: DecodeWorkload) -> dict:
    """Draw Q [B, H, Nq, d] and the cache K, V [B, Hkv, Nk, d], N(0,1), rounded to ``w.dtype``."""
    rng = np.random.Generator(np.random.PCG64(w.seed))
    out = {}
    for name, shape in (("q", (w.B, w.H, w.Nq, w.d)), ("k", (w.B, w.Hkv, w.Nk, w.d)), ("v", (w.B, w.Hkv, w.Nk, w.d))):
        out[name] = round_to_dtype(rng.standard_normal(shape, dtype=np.float32), w.dtype)
    return out


def attention_flops(B, H, N, d, causal, pass_="fwd"):
    """FLOP convention of the metric: forward 4·B·H·N²·d, backward 2.5× that, both halved when causal.

    The forward counts the two N×N×d contractions (2·N²·d each); the backward's
    2.5× counts five contractions including the recomputation of S.
    """
    f = 4.0 * B * H * N * N * d
    if pass_ == "bwd":
        f *= 2.5
    elif pass_ == "fwd+bwd":
        f *= 3.5
    elif pass_ != "fwd":
        raise ValueError(pass_)
    return f / 2.0 if causal else f
