"""Block-sparse and sliding-window attention masks (test infrastructure only).

"Lecture 8 · GPU Performance & FlashAttention" §5.7: block-sparse FlashAttention computes only
a subset of the B_r x B_c blocks of S, so reads, writes and FLOPs fall in proportion to the
non-zero blocks (Proposition 4); the causal mask is the simplest such pattern, and local
windows plus a few global blocks are the general sparse patterns; the sliding window itself
is the approximation the same section measures.  Readings used here (the page gives no
formulas):

* visibility of key j to query i is the conjunction of
  - the block mask: byte [i // 128, j // 128] non-zero (blocks of 128 x 128 scores, the tiles
    the kernels use; one mask per head, or one shared by all heads),
  - causal: j <= i,
  - a window of w > 0: |i - j| < w (with causal: the last w positions up to and including i);
* masked scores are -inf; a row that sees no key has O = 0 and L = -inf, and contributes
  nothing to any gradient.

``attn_fwd64_masked`` / ``attn_bwd64_masked`` are the definition with an explicit boolean
mask; ``tiled_fwd_block_sparse`` follows the method: the FA2-order tiled forward that never
touches a block whose mask is zero, counting the blocks it visits.
"""

from __future__ import annotations

import numpy as np

__all__ = ["visible_mask", "visible_row", "attn_fwd64_masked", "attn_bwd64_masked", "attn_fwd64_masked_rows",
           "tiled_fwd_block_sparse", "blocks_visited", "BLOCK"]

BLOCK = 128


def visible_mask(n, causal=False, window=0, block_mask=None, block=BLOCK):
    """Boolean [N, N] (or [Hm, N, N] for a per-head block mask [Hm, nb, nb]): True where visible."""
    i = np.arange(n)[:, None]
    j = np.arange(n)[None, :]
    vis = np.ones((n, n), dtype=bool)
    if causal:
        vis &= j <= i
    if window and window > 0:
        vis &= np.abs(i - j) < window
    if block_mask is None:
        return vis
    bm = np.asarray(block_mask) != 0
    expand = bm[..., i // block, j // block]  # [..., N, N]
    return vis & expand


def _rows_probabilities(q_rows, k, scale, vis_rows):
    s = scale * (np.asarray(q_rows, np.float64) @ np.asarray(k, np.float64).T)
    s = np.where(vis_rows, s, -np.inf)
    m = s.max(axis=1)
    finite = np.isfinite(m)
    m_safe = np.where(finite, m, 0.0)
    e = np.exp(s - m_safe[:, None])
    ell = e.sum(axis=1)
    p = np.where(finite[:, None], e / np.where(ell > 0, ell, 1.0)[:, None], 0.0)
    with np.errstate(divide="ignore"):
        lse = np.where(finite, m + np.log(np.where(ell > 0, ell, 1.0)), -np.inf)
    return p, lse


def _vis_for(visible, h):
    v = np.asarray(visible)
    return v if v.ndim == 2 else v[h if v.shape[0] > 1 else 0]


def attn_fwd64_masked(q, k, v, scale, visible):
    """O [B, H, N, dv], L [B, H, N] of attention with the boolean mask ``visible`` ([N, N] or [Hm, N, N])."""
    q, k, v = (np.asarray(t, np.float64) for t in (q, k, v))
    b_, h_, n, _ = q.shape
    o = np.zeros((b_, h_, n, v.shape[-1]))
    lse = np.zeros((b_, h_, n))
    for b in range(b_):
        for h in range(h_):
            p, lse[b, h] = _rows_probabilities(q[b, h], k[b, h], scale, _vis_for(visible, h))
            o[b, h] = p @ v[b, h]
    return o, lse


def attn_bwd64_masked(q, k, v, do, scale, visible):
    """dQ, dK, dV of f = sum O*dO for masked attention (masked probabilities are exactly 0)."""
    q, k, v, do = (np.asarray(t, np.float64) for t in (q, k, v, do))
    b_, h_, n, _ = q.shape
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    for b in range(b_):
        for h in range(h_):
            p, _ = _rows_probabilities(q[b, h], k[b, h], scale, _vis_for(visible, h))
            dv[b, h] = p.T @ do[b, h]
            dp = do[b, h] @ v[b, h].T
            d_i = (p * dp).sum(axis=1)
            ds = p * (dp - d_i[:, None])
            dq[b, h] = scale * (ds @ k[b, h])
            dk[b, h] = scale * (ds.T @ q[b, h])
    return dq, dk, dv


def blocks_visited(n, causal=False, window=0, block_mask=None, block=BLOCK):
    """Per head: the (query block, key block) pairs with at least one visible score."""
    vis = visible_mask(n, causal, window, block_mask, block)
    nb = (n + block - 1) // block
    vis = vis if vis.ndim == 3 else vis[None]
    out = np.zeros((vis.shape[0], nb, nb), dtype=bool)
    for a in range(nb):
        for c in range(nb):
            out[:, a, c] = vis[:, a * block:(a + 1) * block, c * block:(c + 1) * block].any(axis=(1, 2))
    return out


def tiled_fwd_block_sparse(q, k, v, scale, visible, block=BLOCK):
    """FA2-order tiled forward of one head (q, k, v: [N, d]) that skips every block of S with no
    visible score; within a visited block masked scores are -inf.  Each visited block updates
    the row state (m, l, O) with the online-softmax rule.  Returns O, L and the number of blocks
    visited."""
    q, k, v = (np.asarray(t, np.float64) for t in (q, k, v))
    vis = np.asarray(visible, dtype=bool)
    n = q.shape[0]
    o = np.zeros((n, v.shape[1]))
    lse = np.full(n, -np.inf)
    visited = 0
    for r0 in range(0, n, block):
        rows = slice(r0, min(n, r0 + block))
        m = np.full(rows.stop - r0, -np.inf)
        ell = np.zeros(rows.stop - r0)
        acc = np.zeros((rows.stop - r0, v.shape[1]))
        for c0 in range(0, n, block):
            cols = slice(c0, min(n, c0 + block))
            vblk = vis[rows, cols]
            if not vblk.any():
                continue  # never loaded, never multiplied
            visited += 1
            s = np.where(vblk, scale * (q[rows] @ k[cols].T), -np.inf)
            m_new = np.maximum(m, s.max(axis=1))
            safe = np.where(np.isfinite(m_new), m_new, 0.0)
            alpha = np.where(np.isfinite(m), np.exp(m - safe), 0.0)
            pt = np.exp(s - safe[:, None])
            ell = alpha * ell + pt.sum(axis=1)
            acc = alpha[:, None] * acc + pt @ v[cols]
            m = m_new
        seen = ell > 0
        o[rows] = np.where(seen[:, None], acc / np.where(seen, ell, 1.0)[:, None], 0.0)
        with np.errstate(divide="ignore"):
            lse[rows] = np.where(seen, m + np.log(np.where(seen, ell, 1.0)), -np.inf)
    return o, lse, visited


def visible_row(n, i, causal=False, window=0, block_mask=None, block=BLOCK):
    """Row i of ``visible_mask`` (block_mask: the head's [nb, nb] mask or None), without the N x N array."""
    j = np.arange(n)
    vis = np.ones(n, dtype=bool)
    if causal:
        vis &= j <= i
    if window and window > 0:
        vis &= np.abs(i - j) < window
    if block_mask is not None:
        vis &= np.asarray(block_mask)[i // block, j // block] != 0
    return vis


def attn_fwd64_masked_rows(q, k, v, scale, samples, causal=False, window=0, block_mask=None, block=BLOCK):
    """O rows [S, dv] and L [S] for sampled (b, h, i) of masked attention (block_mask [nb, nb] or [H, nb, nb])."""
    out_o = np.zeros((len(samples), np.asarray(v).shape[-1]))
    out_l = np.zeros(len(samples))
    n = np.asarray(k).shape[2]
    for t, (b, h, i) in enumerate(samples):
        bm = None
        if block_mask is not None:
            bm = np.asarray(block_mask)
            bm = bm if bm.ndim == 2 else bm[h if bm.shape[0] > 1 else 0]
        vis = visible_row(n, i, causal, window, bm, block)
        p, lse = _rows_probabilities(np.asarray(q[b, h, i], np.float64)[None], k[b, h], scale, vis[None])
        out_o[t] = p[0] @ np.asarray(v[b, h], np.float64)
        out_l[t] = lse[0]
    return out_o, out_l
