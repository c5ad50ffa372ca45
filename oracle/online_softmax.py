"""The method's own steps in fp64: online softmax, state merge, tiled forward and backward.

Test infrastructure only (see ``oracle/__init__.py``).

These functions follow the pages' algorithms step by step, in their order and
notation, with numpy matrix products as the only library primitive.  They are
used to pin the oracle (the tiled method must equal the definition in
``attention.py`` to fp64 rounding, "Lecture 8 · GPU Performance &
FlashAttention" §5.3 and §5.4 report 1e-16…1e-15) and to fix the tile-count
invariant of causal block skipping (§5.7).
"""

from __future__ import annotations

import math

import numpy as np

__all__ = [
    "online_softmax_trace",
    "merge_states",
    "tiled_fwd_fa2_order",
    "tiled_fwd_fa1_order",
    "tiled_bwd_recompute",
    "causal_tiles_visited",
]


def online_softmax_trace(x, block):
    """Online softmax over a stream read ``block`` values at a time.

    "Lecture 8 · GPU Performance & FlashAttention" §5.2: keep the running
    maximum m and the denominator ℓ relative to m; on a new block,
    m_new = max(m, max(block)), ℓ ← ℓ·e^(m − m_new) + Σ e^(x − m_new).
    (Same update, element at a time, in "Stanford CS336 Lecture 5 close
    reading", §7.)  Returns the list of (count_read, m, ℓ) after each block.
    """
    m = -math.inf
    ell = 0.0
    trace = []
    x = [float(t) for t in x]
    for s in range(0, len(x), block):
        blk = x[s:s + block]
        m_new = max(m, max(blk))
        ell = ell * math.exp(m - m_new) + sum(math.exp(t - m_new) for t in blk)
        m = m_new
        trace.append((s + len(blk), m, ell))
    return trace


def merge_states(m1, l1, m2, l2, o1=None, o2=None):
    """Merge two partial online-softmax states (Exercise 3 of the Lecture 8 notes).

    m = max(m1, m2), ℓ = ℓ1·e^(m1−m) + ℓ2·e^(m2−m).  If normalised partial
    outputs o1, o2 are given, the merged output is
    (ℓ1 e^(m1−m) o1 + ℓ2 e^(m2−m) o2) / ℓ (the same rescaling applied to the
    outputs, as Flash-Decoding uses it, §8.2).
    """
    m = max(m1, m2)
    w1 = l1 * math.exp(m1 - m) if math.isfinite(m1) else 0.0
    w2 = l2 * math.exp(m2 - m) if math.isfinite(m2) else 0.0
    ell = w1 + w2
    if o1 is None:
        return m, ell
    o = (w1 * np.asarray(o1, dtype=np.float64) + w2 * np.asarray(o2, dtype=np.float64)) / ell
    return m, ell, o


def _block_causal_skip(r0, c0):
    """Key block starting at c0 lies wholly in the future of query block starting at r0's last row?"""
    return c0 > r0


def tiled_fwd_fa2_order(q, k, v, scale, causal, br, bc, count=None):
    """Tiled exact forward, FA2 loop order, one head: q, k, v [N, d] → (O, L).

    Outer loop over query blocks, inner over key/value blocks; the output is
    kept unnormalised and divided by ℓ once at the end ("Lecture 8" §8.1;
    the loop of "Stanford CS336 Lecture 5 close reading" §7):

        S = τ Q_i K_jᵀ;  m_new = max(m, rowmax S);  P = exp(S − m_new)
        ℓ = ℓ·e^(m − m_new) + rowsum P;  O = O·e^(m − m_new) + P V_j;  m = m_new
        after the last block: O = O / ℓ,  L = m + ln ℓ.

    Under the causal mask, key blocks wholly in the future of the query block
    are neither read nor computed (§5.3 closing paragraph); ``count`` (a list)
    receives the number of visited (i, j) block pairs.
    """
    q, k, v = (np.asarray(t, dtype=np.float64) for t in (q, k, v))
    n, d = q.shape
    o_out = np.zeros((n, d))
    l_out = np.zeros(n)
    visited = 0
    for r0 in range(0, n, br):
        r1 = min(n, r0 + br)
        qi = q[r0:r1]
        m = np.full(r1 - r0, -np.inf)
        ell = np.zeros(r1 - r0)
        o = np.zeros((r1 - r0, d))
        for c0 in range(0, n, bc):
            c1 = min(n, c0 + bc)
            if causal and _block_causal_skip(r1 - 1, c0):
                continue
            visited += 1
            s = scale * (qi @ k[c0:c1].T)
            if causal:
                s = np.where(np.arange(c0, c1)[None, :] > np.arange(r0, r1)[:, None], -np.inf, s)
            m_new = np.maximum(m, s.max(axis=1))
            # rows whose scores so far are all masked keep a −∞ maximum
            m_ref = np.where(np.isfinite(m_new), m_new, 0.0)
            p = np.exp(s - m_ref[:, None])
            alpha = np.where(np.isfinite(m), np.exp(m - m_ref), 0.0)
            ell = ell * alpha + p.sum(axis=1)
            o = o * alpha[:, None] + p @ v[c0:c1]
            m = m_new
        with np.errstate(divide="ignore", invalid="ignore"):
            o_out[r0:r1] = np.where(ell[:, None] > 0, o / np.where(ell > 0, ell, 1.0)[:, None], 0.0)
            l_out[r0:r1] = np.where(ell > 0, m + np.log(np.where(ell > 0, ell, 1.0)), -np.inf)
    if count is not None:
        count.append(visited)
    return o_out, l_out


def tiled_fwd_fa1_order(q, k, v, scale, causal, br, bc):
    """Tiled exact forward, FA1 loop order (Algorithm 1 of "Lecture 8" §5.3), one head.

    Outer loop over key/value blocks, inner over query blocks; O_i, ℓ_i, m_i
    live "in HBM" (here: arrays) between visits and O_i is kept normalised:

        S = τ Q_i K_jᵀ;  m̃ = rowmax S;  P̃ = exp(S − m̃);  ℓ̃ = rowsum P̃
        m_new = max(m_i, m̃);  ℓ_new = e^(m_i − m_new) ℓ_i + e^(m̃ − m_new) ℓ̃
        O_i ← diag(ℓ_new)⁻¹ (diag(ℓ_i) e^(m_i − m_new) O_i + e^(m̃ − m_new) P̃ V_j)

    Returns (O, L) like ``tiled_fwd_fa2_order``.
    """
    q, k, v = (np.asarray(t, dtype=np.float64) for t in (q, k, v))
    n, d = q.shape
    o = np.zeros((n, d))
    ell = np.zeros(n)
    m = np.full(n, -np.inf)
    for c0 in range(0, n, bc):
        c1 = min(n, c0 + bc)
        for r0 in range(0, n, br):
            r1 = min(n, r0 + br)
            if causal and _block_causal_skip(r1 - 1, c0):
                continue
            s = scale * (q[r0:r1] @ k[c0:c1].T)
            if causal:
                s = np.where(np.arange(c0, c1)[None, :] > np.arange(r0, r1)[:, None], -np.inf, s)
            m_t = s.max(axis=1)
            fin_t = np.isfinite(m_t)
            p_t = np.exp(s - np.where(fin_t, m_t, 0.0)[:, None])
            l_t = p_t.sum(axis=1)
            m_i, l_i, o_i = m[r0:r1], ell[r0:r1], o[r0:r1]
            m_new = np.maximum(m_i, m_t)
            fin_new = np.isfinite(m_new)
            m_ref = np.where(fin_new, m_new, 0.0)
            a_old = np.where(np.isfinite(m_i), np.exp(m_i - m_ref), 0.0)
            a_new = np.where(fin_t, np.exp(m_t - m_ref), 0.0)
            l_new = a_old * l_i + a_new * l_t
            safe = np.where(l_new > 0, l_new, 1.0)
            o[r0:r1] = np.where(
                (l_new > 0)[:, None],
                ((l_i * a_old)[:, None] * o_i + a_new[:, None] * (p_t @ v[c0:c1])) / safe[:, None],
                0.0,
            )
            ell[r0:r1] = l_new
            m[r0:r1] = m_new
    with np.errstate(divide="ignore"):
        lse = np.where(ell > 0, m + np.log(np.where(ell > 0, ell, 1.0)), -np.inf)
    return o, lse


def tiled_bwd_recompute(q, k, v, o, do, lse, scale, causal, br, bc):
    """Block-wise backward with recomputation, one head ("Lecture 8" §5.4).

    Nothing N×N is stored: for every visited block pair the scores and
    probabilities are recomputed from Q, K and the row statistic L
    (P_ij = e^(S_ij − m_i)/ℓ_i = e^(S_ij − L_i)), and D_i = Σ_k dO_ik O_ik
    replaces the N×N reduction.  Per block pair (i, j):

        S = τ Q_i K_jᵀ;  P = exp(S − L_i);  dV_j += Pᵀ dO_i;  dP = dO_i V_jᵀ
        dS = P ∘ (dP − D_i);  dK_j += τ dSᵀ Q_i;  dQ_i += τ dS K_j

    Returns dQ, dK, dV [N, d] in fp64.
    """
    q, k, v, o, do, lse = (np.asarray(t, dtype=np.float64) for t in (q, k, v, o, do, lse))
    n, d = q.shape
    d_row = (do * o).sum(axis=1)
    dq = np.zeros((n, d))
    dk = np.zeros((n, d))
    dv = np.zeros((n, d))
    for c0 in range(0, n, bc):
        c1 = min(n, c0 + bc)
        for r0 in range(0, n, br):
            r1 = min(n, r0 + br)
            if causal and _block_causal_skip(r1 - 1, c0):
                continue
            s = scale * (q[r0:r1] @ k[c0:c1].T)
            if causal:
                s = np.where(np.arange(c0, c1)[None, :] > np.arange(r0, r1)[:, None], -np.inf, s)
            li = lse[r0:r1]
            p = np.where(np.isfinite(li)[:, None], np.exp(s - np.where(np.isfinite(li), li, 0.0)[:, None]), 0.0)
            dv[c0:c1] += p.T @ do[r0:r1]
            dp = do[r0:r1] @ v[c0:c1].T
            ds = p * (dp - d_row[r0:r1, None])
            dk[c0:c1] += scale * (ds.T @ q[r0:r1])
            dq[r0:r1] += scale * (ds @ k[c0:c1])
    return dq, dk, dv


def causal_tiles_visited(n, br, bc):
    """Number of (query block, key block) pairs a causal tiled pass visits.

    A key block is skipped when all of its keys lie in the future of every row
    of the query block ("Lecture 8" §5.3 closing paragraph, §5.7).
    """
    total = 0
    for r0 in range(0, n, br):
        r_last = min(n, r0 + br) - 1
        for c0 in range(0, n, bc):
            if not _block_causal_skip(r_last, c0):
                total += 1
    return total
