"""Grouped-query / multi-query attention in fp64 (test infrastructure only, see oracle/__init__.py).

"Lecture 8 · GPU Performance & FlashAttention" §8.2: in MQA and GQA several query heads share
one key/value head, which shrinks the KV cache.  With H query heads and H_kv key/value heads
(H a multiple of H_kv, group size g = H / H_kv), query head h of a batch row reads key/value
head h // g of the same batch row.  Written out from that definition:

* forward: ordinary attention per query head with the K, V of its key/value head;
* backward: the shared K and V receive the sum of the gradients of every query head that
  reads them (the chain rule for a parameter used g times).
"""

from __future__ import annotations

import numpy as np

from .attention import attn_bwd64, attn_fwd64

__all__ = ["kv_head_of", "expand_kv", "attn_fwd64_gqa", "attn_bwd64_gqa"]


def kv_head_of(h: int, n_heads: int, n_kv_heads: int) -> int:
    """Key/value head read by query head h."""
    if n_heads % n_kv_heads:
        raise ValueError("the number of query heads must be a multiple of the key/value heads")
    return h // (n_heads // n_kv_heads)


def expand_kv(x, n_heads: int):
    """[B, H_kv, N, d] -> [B, H, N, d]: each key/value head repeated for its g query heads."""
    x = np.asarray(x, dtype=np.float64)
    g = n_heads // x.shape[1]
    return np.repeat(x, g, axis=1)


def attn_fwd64_gqa(q, k, v, scale, causal=False):
    """O [B, H, N, d] and L [B, H, N] for q [B, H, N, d] and k, v [B, H_kv, N, d]."""
    h = q.shape[1]
    return attn_fwd64(q, expand_kv(k, h), expand_kv(v, h), scale, causal)


def attn_bwd64_gqa(q, k, v, do, scale, causal=False):
    """dQ [B, H, N, d], dK, dV [B, H_kv, N, d] and D [B, H, N] of f = sum(O o dO)."""
    b, h, n, d = q.shape
    h_kv = k.shape[1]
    dq, dk_e, dv_e, dd = attn_bwd64(q, expand_kv(k, h), expand_kv(v, h), do, scale, causal)
    g = h // h_kv
    dk = dk_e.reshape(b, h_kv, g, n, d).sum(axis=2)
    dv = dv_e.reshape(b, h_kv, g, n, dv_e.shape[-1]).sum(axis=2)
    return dq, dk, dv, dd
