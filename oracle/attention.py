"""Standard (materialising) attention in fp64: the definition the method must reproduce.

Test infrastructure only (see ``oracle/__init__.py``): never imported by the
product path.

The exact result the tiled method reaches is plain scaled-dot-product
attention ("Lecture 8 · GPU Performance & FlashAttention", §5.1, the three-step
"Algorithm 0": S = τ·Q·Kᵀ, P = softmax(S), O = P·V), computed with the
safe-softmax convention of the same section (subtract the row maximum before
exponentiating).  The per-row statistic kept for the backward pass is the
log-sum-exp L_i = m_i + ln ℓ_i (§5.4: only O and the two row statistics m, ℓ
are stored; L combines them into one number, natural-log units).

Causal masking: row i sees keys j ≤ i (top-left aligned, queries and keys of
equal length), masked scores are −∞ (§5.3 closing paragraph).  A row with no
visible key (impossible for the square top-left mask used here) yields O = 0
and L = −∞.

The backward pass is the analytic gradient of f = Σ O∘dO, written out from the
definition (§5.4; the printed equations were lost in extraction, the surviving
D identity fixes their form):

    dV = Pᵀ dO
    dP = dO Vᵀ
    D_i = Σ_j P_ij dP_ij          (equal to Σ_k dO_ik O_ik, §5.4)
    dS = P ∘ (dP − D 1ᵀ)
    dQ = τ dS K
    dK = τ dSᵀ Q

All arrays are numpy, layout [B, H, N, d] (one N×d matrix per head, §5.1),
row statistics [B, H, N].  S and P are materialised one block of query rows
at a time; every row's softmax still spans the whole row, so this is the
standard algorithm, only with bounded memory.
"""

from __future__ import annotations

import numpy as np

__all__ = [
    "probabilities64",
    "attn_fwd64",
    "attn_bwd64",
    "attn_fwd64_rows",
    "attn_bwd64_query_rows",
    "attn_stats64",
    "attn_bwd64_key_rows",
]

# Query rows materialised at once per head (bounds the S/P block to rows × N).
_ROW_BLOCK = 1024


def _f64(x):
    return np.asarray(x, dtype=np.float64)


def _causal_mask(row_idx: np.ndarray, n_keys: int) -> np.ndarray:
    """True where key j is in the future of query row i (j > i)."""
    return np.arange(n_keys)[None, :] > row_idx[:, None]


def probabilities64(q_rows, k, scale, causal, row_idx):
    """Rows of S and P for the given query rows of one head.

    q_rows: [R, d] query rows; k: [N, d]; row_idx: the rows' positions (for the
    causal mask).  Returns (S, P, m, ell) with S, P: [R, N] and m, ell: [R].
    Masked scores are −∞ and their probabilities exactly 0.
    """
    q_rows = _f64(q_rows)
    k = _f64(k)
    s = scale * (q_rows @ k.T)
    if causal:
        s = np.where(_causal_mask(np.asarray(row_idx), k.shape[0]), -np.inf, s)
    m = s.max(axis=1)
    finite = np.isfinite(m)
    m_safe = np.where(finite, m, 0.0)
    e = np.exp(s - m_safe[:, None])  # exp(−∞) = 0 for masked entries
    ell = e.sum(axis=1)
    p = np.where(finite[:, None], e / np.where(ell > 0, ell, 1.0)[:, None], 0.0)
    return s, p, m, ell


def _lse(m, ell):
    with np.errstate(divide="ignore"):
        return np.where(np.isfinite(m), m + np.log(ell), -np.inf)


def attn_fwd64(q, k, v, scale, causal=False):
    """Forward pass: O = softmax(τ Q Kᵀ [+ mask]) V and L = rowwise log-sum-exp.

    q, k, v: [B, H, N, d] (any float dtype; computed in fp64).
    Returns O [B, H, N, d] fp64 and L [B, H, N] fp64.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    b_, h_, n, _ = q.shape
    o = np.zeros((b_, h_, n, v.shape[-1]))
    lse = np.zeros((b_, h_, n))
    for b in range(b_):
        for h in range(h_):
            for r0 in range(0, n, _ROW_BLOCK):
                rows = np.arange(r0, min(n, r0 + _ROW_BLOCK))
                _, p, m, ell = probabilities64(q[b, h, rows], k[b, h], scale, causal, rows)
                o[b, h, rows] = p @ v[b, h]
                lse[b, h, rows] = _lse(m, ell)
    return o, lse


def attn_bwd64(q, k, v, do, scale, causal=False):
    """Backward pass of f = Σ O∘dO from the definition (P recomputed exactly).

    Returns dQ, dK, dV [B, H, N, d] and D [B, H, N] (D_i = Σ_j P_ij dP_ij), all fp64.
    """
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    b_, h_, n, d = q.shape
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    dd = np.zeros((b_, h_, n))
    for b in range(b_):
        for h in range(h_):
            for r0 in range(0, n, _ROW_BLOCK):
                rows = np.arange(r0, min(n, r0 + _ROW_BLOCK))
                _, p, _, _ = probabilities64(q[b, h, rows], k[b, h], scale, causal, rows)
                do_r = do[b, h, rows]
                dv[b, h] += p.T @ do_r
                dp = do_r @ v[b, h].T
                d_i = (p * dp).sum(axis=1)
                ds = p * (dp - d_i[:, None])
                dq[b, h, rows] = scale * (ds @ k[b, h])
                dk[b, h] += scale * (ds.T @ q[b, h, rows])
                dd[b, h, rows] = d_i
    return dq, dk, dv, dd


# ---------------------------------------------------------------------------
# Sampled paths: exact per-row (or per-key) results for problems too large to
# materialise whole.  Each sampled output is still the plain definition.
# ---------------------------------------------------------------------------


def attn_fwd64_rows(q, k, v, scale, causal, samples):
    """O rows and L values for sampled (b, h, i) triples.

    samples: int array [S, 3].  Row i of O needs q_i and all of K, V only.
    Returns O [S, d] and L [S] in fp64.
    """
    samples = np.asarray(samples, dtype=np.int64)
    o = np.zeros((len(samples), v.shape[-1]))
    lse = np.zeros(len(samples))
    for t, (b, h, i) in enumerate(samples):
        _, p, m, ell = probabilities64(_f64(q[b, h, i])[None, :], k[b, h], scale, causal, np.array([i]))
        o[t] = p[0] @ _f64(v[b, h])
        lse[t] = _lse(m, ell)[0]
    return o, lse


def attn_bwd64_query_rows(q, k, v, do, scale, causal, samples):
    """dQ rows (and D_i) for sampled (b, h, i) triples, exact per row.

    dQ_i = τ Σ_j P_ij (dP_ij − D_i) K_j with dP_ij = dO_i·V_j and D_i = Σ_j P_ij dP_ij:
    row i's own P and dP suffice.
    """
    samples = np.asarray(samples, dtype=np.int64)
    d = q.shape[-1]
    dq = np.zeros((len(samples), d))
    dd = np.zeros(len(samples))
    for t, (b, h, i) in enumerate(samples):
        kk = _f64(k[b, h])
        _, p, _, _ = probabilities64(_f64(q[b, h, i])[None, :], kk, scale, causal, np.array([i]))
        dp = _f64(v[b, h]) @ _f64(do[b, h, i])
        d_i = float(p[0] @ dp)
        dq[t] = scale * ((p[0] * (dp - d_i)) @ kk)
        dd[t] = d_i
    return dq, dd


def attn_stats64(q, k, v, do, scale, causal, b, h):
    """All rows' L_i and D_i of one head, streaming S, P one row block at a time.

    Needed by the key-side sampled gradients: column j of P involves every row's
    normalisation.  Returns (L [N], D [N]) in fp64.
    """
    n = q.shape[2]
    kk, vv = _f64(k[b, h]), _f64(v[b, h])
    lse = np.zeros(n)
    dd = np.zeros(n)
    for r0 in range(0, n, _ROW_BLOCK):
        rows = np.arange(r0, min(n, r0 + _ROW_BLOCK))
        _, p, m, ell = probabilities64(_f64(q[b, h, rows]), kk, scale, causal, rows)
        dp = _f64(do[b, h, rows]) @ vv.T
        lse[rows] = _lse(m, ell)
        dd[rows] = (p * dp).sum(axis=1)
    return lse, dd


def attn_bwd64_key_rows(q, k, v, do, scale, causal, b, h, keys, stats=None):
    """dK_j and dV_j for sampled key rows j of head (b, h), exact.

    dV_j = Σ_i P_ij dO_i and dK_j = τ Σ_i P_ij (dP_ij − D_i) Q_i, with
    P_ij = exp(S_ij − L_i).  ``stats`` may pass precomputed (L, D) of that head
    from ``attn_stats64``.  Returns dK [len(keys), d], dV [len(keys), d].
    """
    keys = np.asarray(keys, dtype=np.int64)
    if stats is None:
        stats = attn_stats64(q, k, v, do, scale, causal, b, h)
    lse, dd = stats
    qq, dOo = _f64(q[b, h]), _f64(do[b, h])
    kj, vj = _f64(k[b, h, keys]), _f64(v[b, h, keys])
    s = scale * (qq @ kj.T)  # [N, J]: column t is key keys[t]
    if causal:
        s = np.where(np.arange(qq.shape[0])[:, None] < keys[None, :], -np.inf, s)
    with np.errstate(invalid="ignore"):
        p = np.where(np.isfinite(lse)[:, None], np.exp(s - lse[:, None]), 0.0)
    dp = dOo @ vj.T
    ds = p * (dp - dd[:, None])
    dv = p.T @ dOo
    dk = scale * (ds.T @ qq)
    return dk, dv
