"""Decode-time attention over a long key/value cache, and its split-KV form (test infrastructure only).

"Lecture 8 · GPU Performance & FlashAttention" §8.2: when a few queries attend to a very long
KV cache, the cache is cut into pieces processed in parallel and the partial results are
combined with the merge formula of the online softmax (Exercise 3: m = max(m1, m2),
ℓ = ℓ1 e^(m1−m) + ℓ2 e^(m2−m), with the same rescaling applied to the outputs).

Shapes: Q [B, H, Nq, d] (the new queries), K, V [B, H_kv, Nk, d] (the cache, H a multiple of
H_kv), every query sees every cached key (no mask: the queries are the latest positions).

* ``decode_fwd64`` is the definition: attention of each query row over all Nk keys.
* ``split_kv_states64`` follows the method: per split, the partial state (m, ℓ, O normalised
  within the split) from the definition restricted to that split's keys; ``merge_splits64``
  then folds the splits with ``merge_states`` in order.
"""

from __future__ import annotations

import numpy as np

from .attention import probabilities64
from .gqa import expand_kv
from .online_softmax import merge_states

__all__ = ["decode_fwd64", "split_kv_states64", "merge_splits64", "split_bounds"]


def decode_fwd64(q, k, v, scale):
    """O [B, H, Nq, d] and L [B, H, Nq] of every query row over the whole cache."""
    q = np.asarray(q, dtype=np.float64)
    b_, h_, nq, _ = q.shape
    ke, ve = expand_kv(k, h_), expand_kv(v, h_)
    o = np.zeros((b_, h_, nq, ve.shape[-1]))
    lse = np.zeros((b_, h_, nq))
    for b in range(b_):
        for h in range(h_):
            _, p, m, ell = probabilities64(q[b, h], ke[b, h], scale, False, np.arange(nq))
            o[b, h] = p @ ve[b, h]
            lse[b, h] = m + np.log(ell)
    return o, lse


def split_bounds(nk, splits):
    """Key ranges [start, end) of `splits` consecutive pieces of the cache, as equal as possible."""
    edges = [(nk * s) // splits for s in range(splits + 1)]
    return [(edges[s], edges[s + 1]) for s in range(splits)]


def split_kv_states64(q, k, v, scale, splits):
    """Per split: m [B, H, Nq], ℓ [B, H, Nq] and O normalised within the split [B, H, Nq, d].

    An empty split has m = −∞, ℓ = 0 and O = 0 (it contributes nothing to the merge).
    """
    q = np.asarray(q, dtype=np.float64)
    b_, h_, nq, _ = q.shape
    ke, ve = expand_kv(k, h_), expand_kv(v, h_)
    states = []
    for lo, hi in split_bounds(ke.shape[2], splits):
        m = np.full((b_, h_, nq), -np.inf)
        ell = np.zeros((b_, h_, nq))
        o = np.zeros((b_, h_, nq, ve.shape[-1]))
        if hi > lo:
            for b in range(b_):
                for h in range(h_):
                    _, p, mm, ll = probabilities64(q[b, h], ke[b, h, lo:hi], scale, False, np.arange(nq))
                    m[b, h], ell[b, h] = mm, ll
                    o[b, h] = p @ ve[b, h, lo:hi]
        states.append((m, ell, o))
    return states


def merge_splits64(states):
    """Fold the split states in order with the Exercise 3 merge: returns O and L = m + ln ℓ."""
    m, ell, o = states[0]
    m, ell, o = m.copy(), ell.copy(), o.copy()
    for m2, l2, o2 in states[1:]:
        for idx in np.ndindex(m.shape):
            if not np.isfinite(m2[idx]):
                continue
            if not np.isfinite(m[idx]):
                m[idx], ell[idx], o[idx] = m2[idx], l2[idx], o2[idx]
                continue
            m[idx], ell[idx], o[idx] = merge_states(m[idx], ell[idx], m2[idx], l2[idx], o[idx], o2[idx])
    return o, m + np.log(ell)
