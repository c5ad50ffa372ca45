"""FP8 (E4M3) block quantisation and attention on the dequantised inputs (test infrastructure only).

"Lecture 8 · GPU Performance & FlashAttention" §8.1 and "FlashAttention and GPU memory" §11:
the third generation runs attention in 8-bit floating point with block quantisation (one
scale per block of a tensor rather than one per tensor), which keeps the error well below
that of a per-tensor FP8 baseline.  The pages fix neither the block shape nor the format;
the readings used here:

* format: E4M3 as in the OCP 8-bit floating point specification (1 sign bit, 4 exponent
  bits with bias 7, 3 mantissa bits; subnormals down to 2^-9; largest finite value 448; no
  infinities), rounding to nearest with ties to even, saturating at +-448;
* blocks: for each head, consecutive blocks of 128 rows x all d columns of Q, K and V (the
  tiles the attention kernel streams); the scale of a block is amax / 448 (1 for an all-zero
  block) and its codes are E4M3(x / scale);
* the two decisions that produce codes (the scale and the quotient) are taken in fp32, the
  precision of the quantising kernel, so that codes can be compared bit for bit;
* attention: exact attention (``attn_fwd64``) on the dequantised tensors code x scale.

Everything else is fp64.
"""

from __future__ import annotations

import numpy as np

from .attention import attn_fwd64

__all__ = ["E4M3_MAX", "e4m3_round", "e4m3_values", "quantize_blocks", "dequantize_blocks", "attn_fwd64_fp8"]

E4M3_MAX = 448.0
_MANTISSA_BITS = 3
_MIN_NORMAL_EXP = -6  # 2^(1 - 7)


def e4m3_values() -> np.ndarray:
    """All non-negative finite E4M3 values, ascending (from the format's definition)."""
    vals = [m * 2.0 ** (_MIN_NORMAL_EXP - _MANTISSA_BITS) for m in range(8)]  # subnormals and zero
    for e in range(1, 16):
        for m in range(8):
            if e == 15 and m == 7:
                continue  # S.1111.111 is NaN
            vals.append((1 + m / 8.0) * 2.0 ** (e - 7))
    return np.array(vals)


def e4m3_round(x) -> np.ndarray:
    """Round to the nearest E4M3 value, ties to the even mantissa, saturating at +-448."""
    x = np.asarray(x, dtype=np.float64)
    a = np.minimum(np.abs(x), E4M3_MAX)
    # spacing of the representable values around a: 2^(e - 3) for a in [2^e, 2^(e+1)), and the
    # subnormal spacing 2^-9 below the smallest normal 2^-6
    _, fe = np.frexp(np.where(a > 0, a, 1.0))  # a = f 2^fe with f in [0.5, 1): a in [2^(fe-1), 2^fe)
    e = np.maximum(fe - 1, _MIN_NORMAL_EXP).astype(np.float64)
    ulp = 2.0 ** (e - _MANTISSA_BITS)
    q = a / ulp                      # exact: a power-of-two scaling
    r = np.round(q)                  # numpy rounds halves to even
    out = r * ulp
    return np.where(np.signbit(x), -out, out)


def quantize_blocks(x, block: int = 128):
    """Block quantisation of x [..., N, d]: codes (as their float values) and scales [..., ceil(N/block)].

    scale = float32(amax) / float32(448) in fp32, codes = E4M3(float32(x) / scale) with the
    quotient in fp32; amax = 0 gives scale 1.
    """
    x32 = np.asarray(x, dtype=np.float32)
    n = x32.shape[-2]
    nb = (n + block - 1) // block
    scales = np.empty(x32.shape[:-2] + (nb,), dtype=np.float32)
    codes = np.empty(x32.shape, dtype=np.float64)
    for b in range(nb):
        blk = x32[..., b * block:(b + 1) * block, :]
        amax = np.abs(blk).max(axis=(-2, -1)).astype(np.float32)
        s = np.where(amax > 0, amax / np.float32(E4M3_MAX), np.float32(1.0)).astype(np.float32)
        scales[..., b] = s
        quot = (blk / s[..., None, None]).astype(np.float32)
        codes[..., b * block:(b + 1) * block, :] = e4m3_round(quot)
    return codes, scales


def dequantize_blocks(codes, scales, block: int = 128):
    """code x scale of its block, in fp64."""
    codes = np.asarray(codes, dtype=np.float64)
    rep = np.repeat(np.asarray(scales, dtype=np.float64), block, axis=-1)[..., : codes.shape[-2]]
    return codes * rep[..., None]


def attn_fwd64_fp8(q_codes, q_scales, k_codes, k_scales, v_codes, v_scales, scale, causal, block: int = 128):
    """O, L of exact attention on the dequantised Q, K, V."""
    return attn_fwd64(dequantize_blocks(q_codes, q_scales, block), dequantize_blocks(k_codes, k_scales, block),
                      dequantize_blocks(v_codes, v_scales, block), scale, causal)
