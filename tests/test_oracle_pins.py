"""Pins of the fp64 oracle against what the pages and mathematics fix (CPU only).

Each check is chosen so that a plausible slip in the oracle (a dropped term, a
wrong sign or index, a transposed operand) fails at least one of them; the
planted-mistake tests at the end demonstrate that for several such slips.
"""

import math

import numpy as np
import pytest

import oracle
from oracle import attention as A
from oracle import online_softmax as OS
from exact_tiled_attention_07_gb300.inputs import attention_flops

RNG = np.random.default_rng(1234)


def _rand(*shape, rng=RNG):
    return rng.standard_normal(shape)


# --------------------------------------------------------------------------
# values printed on the pages
# --------------------------------------------------------------------------


def test_online_softmax_worked_example(golden):
    kv, rows = golden("online_softmax_worked_example.txt")
    x = kv["x"]
    trace = oracle.online_softmax_trace(x, int(kv["block"][0]))
    assert len(trace) == len(rows)
    for (n_read, m, ell), (g_read, g_m, g_ell) in zip(trace, rows):
        assert n_read == int(g_read)
        assert m == g_m
        assert abs(ell - g_ell) < 5e-7  # the page prints six decimals
    # the final denominator is the whole-row one, exactly up to rounding
    assert abs(trace[-1][2] - sum(math.exp(t - 6.0) for t in x)) < 1e-15


def test_merge_exercise3(golden):
    kv, _ = golden("merge_exercise3.txt")
    (_, m1, l1), = oracle.online_softmax_trace(kv["x1"], 2)
    (_, m2, l2), = oracle.online_softmax_trace(kv["x2"], 2)
    assert (m1, round(l1, 6)) == tuple(kv["state1"])
    assert (m2, round(l2, 6)) == tuple(kv["state2"])
    m, ell = oracle.merge_states(m1, l1, m2, l2)
    assert (m, round(ell, 6)) == tuple(kv["merged"])
    # merged state equals the state of the concatenated stream
    (_, md, ld), = oracle.online_softmax_trace(kv["x1"] + kv["x2"], 4)
    assert m == md and abs(ell - ld) < 1e-15


def test_merge_outputs_equal_whole_row():
    # merging two normalised partial outputs reproduces softmax-weighted sums of the whole row
    s = _rand(10) * 3
    v = _rand(10, 4)
    def part(lo, hi):
        m = s[lo:hi].max()
        e = np.exp(s[lo:hi] - m)
        return m, e.sum(), (e @ v[lo:hi]) / e.sum()
    m1, l1, o1 = part(0, 6)
    m2, l2, o2 = part(6, 10)
    _, _, o = oracle.merge_states(m1, l1, m2, l2, o1, o2)
    p = np.exp(s - s.max()); p /= p.sum()
    np.testing.assert_allclose(o, p @ v, atol=1e-15, rtol=0)


def test_flop_convention_exercise1(golden):
    kv, _ = golden("exercise1_qkt_accounting.txt")
    n, d, e = int(kv["N"][0]), int(kv["d"][0]), int(kv["bytes_per_element"][0])
    # the forward counts two N×N×d contractions; one of them is Exercise 1's Q·Kᵀ
    assert attention_flops(1, 1, n, d, False, "fwd") / 2 == kv["flops"][0]
    qkt_bytes = e * (n * d + d * n + n * n)
    assert qkt_bytes == kv["bytes"][0]
    assert round(kv["flops"][0] / qkt_bytes, 1) == kv["intensity"][0]
    assert attention_flops(2, 3, 128, 64, True, "bwd") == 2.5 * 4 * 6 * 128 * 128 * 64 / 2


def test_causal_tile_count(golden):
    kv, _ = golden("causal_tile_count.txt")
    t = int(kv["blocks_per_side"][0])
    br = 16
    assert oracle.causal_tiles_visited(t * br, br, br) == kv["visited"][0]
    assert round(kv["visited"][0] / kv["total"][0], 3) == kv["fraction"][0]
    # the tiled forward visits exactly that many block pairs
    cnt = []
    q, k, v = _rand(t * br, 4), _rand(t * br, 4), _rand(t * br, 4)
    OS.tiled_fwd_fa2_order(q, k, v, 0.5, True, br, br, count=cnt)
    assert cnt == [136]
    for tt in (1, 2, 7, 32):
        assert oracle.causal_tiles_visited(tt * 128, 128, 128) == tt * (tt + 1) // 2


# --------------------------------------------------------------------------
# the tiled method equals the definition to fp64 rounding
# --------------------------------------------------------------------------


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("br,bc", [(16, 16), (32, 64), (64, 32), (256, 256), (48, 80)])
def test_tiled_forward_equals_standard(causal, br, bc):
    n, d = 256, 32
    rng = np.random.default_rng(7)
    q, k, v = (rng.standard_normal((1, 1, n, d)) for _ in range(3))
    tau = 1 / math.sqrt(d)
    o_ref, l_ref = oracle.attn_fwd64(q, k, v, tau, causal)
    for fn in (OS.tiled_fwd_fa2_order, OS.tiled_fwd_fa1_order):
        o, lse = fn(q[0, 0], k[0, 0], v[0, 0], tau, causal, br, bc)
        assert np.abs(o - o_ref[0, 0]).max() < 5e-15
        assert np.abs(lse - l_ref[0, 0]).max() < 5e-15


@pytest.mark.parametrize("causal", [False, True])
def test_recompute_backward_equals_definition(causal):
    n, d = 160, 16
    rng = np.random.default_rng(9)
    q, k, v, do = (rng.standard_normal((1, 1, n, d)) for _ in range(4))
    tau = 0.3
    o, lse = oracle.attn_fwd64(q, k, v, tau, causal)
    dq, dk, dv, _ = oracle.attn_bwd64(q, k, v, do, tau, causal)
    for br, bc in [(32, 32), (64, 48), (160, 160)]:
        tq, tk, tv = OS.tiled_bwd_recompute(q[0, 0], k[0, 0], v[0, 0], o[0, 0], do[0, 0], lse[0, 0], tau, causal, br, bc)
        for a, b in ((tq, dq), (tk, dk), (tv, dv)):
            assert np.abs(a - b[0, 0]).max() < 1e-13 * max(1.0, np.abs(b).max())


# --------------------------------------------------------------------------
# mathematics: invariants, closed forms, finite differences
# --------------------------------------------------------------------------


@pytest.mark.parametrize("causal", [False, True])
def test_probability_rows(causal):
    q, k = _rand(33, 8), _rand(33, 8)
    _, p, _, _ = A.probabilities64(q, k, 0.7, causal, np.arange(33))
    assert (p >= 0).all()
    np.testing.assert_allclose(p.sum(axis=1), 1.0, atol=1e-15, rtol=0)
    if causal:
        assert (p[np.triu_indices(33, 1)] == 0).all()


def test_single_key_closed_form():
    q, k, v = _rand(2, 3, 1, 5), _rand(2, 3, 1, 5), _rand(2, 3, 1, 5)
    for causal in (False, True):
        o, lse = oracle.attn_fwd64(q, k, v, 0.25, causal)
        np.testing.assert_array_equal(o, v)
        np.testing.assert_allclose(lse, 0.25 * (q * k).sum(-1), atol=1e-15, rtol=0)


def test_equal_keys_give_means():
    n, d = 12, 4
    q = _rand(1, 1, n, d)
    k = np.broadcast_to(_rand(1, 1, 1, d), (1, 1, n, d)).copy()
    v = _rand(1, 1, n, d)
    o, lse = oracle.attn_fwd64(q, k, v, 1.0, False)
    np.testing.assert_allclose(o[0, 0], np.broadcast_to(v[0, 0].mean(0), (n, d)), atol=1e-14)
    np.testing.assert_allclose(lse[0, 0], (q[0, 0] @ k[0, 0, 0]) + math.log(n), atol=1e-14)
    o, lse = oracle.attn_fwd64(q, k, v, 1.0, True)
    prefix = np.cumsum(v[0, 0], axis=0) / np.arange(1, n + 1)[:, None]
    np.testing.assert_allclose(o[0, 0], prefix, atol=1e-14)
    np.testing.assert_allclose(lse[0, 0], (q[0, 0] @ k[0, 0, 0]) + np.log(np.arange(1, n + 1)), atol=1e-14)


def test_constant_values_pass_through():
    q, k = _rand(1, 2, 9, 3), _rand(1, 2, 9, 3)
    v = np.ones((1, 2, 9, 3))
    for causal in (False, True):
        o, _ = oracle.attn_fwd64(q, k, v, 1.3, causal)
        np.testing.assert_allclose(o, 1.0, atol=1e-15, rtol=0)


def test_per_query_shift_invariance():
    # an extra coordinate with q' = c_i / τ and k' = 1 adds c_i to every score of row i
    n, d, tau = 10, 4, 0.5
    q, k, v = _rand(1, 1, n, d), _rand(1, 1, n, d), _rand(1, 1, n, d)
    c = _rand(n) * 5
    q2 = np.concatenate([q, (c / tau)[None, None, :, None]], axis=-1)
    k2 = np.concatenate([k, np.ones((1, 1, n, 1))], axis=-1)
    for causal in (False, True):
        o1, l1 = oracle.attn_fwd64(q, k, v, tau, causal)
        o2, l2 = oracle.attn_fwd64(q2, k2, v, tau, causal)
        np.testing.assert_allclose(o2, o1, atol=1e-14)
        np.testing.assert_allclose(l2 - l1, c[None, None, :], atol=1e-13)


def test_key_offset_moves_probability_mass():
    # a per-key offset c_j (the long-sequence workload's recipe) multiplies column j of e^S by e^(c_j)
    n, d, tau = 8, 3, 0.5
    q, k, v = _rand(1, 1, n, d), _rand(1, 1, n, d), _rand(1, 1, n, d)
    c = _rand(n)
    q2 = np.concatenate([np.ones((1, 1, n, 1)), q], axis=-1)
    k2 = np.concatenate([(c / tau)[None, None, :, None], k], axis=-1)
    _, p1, _, _ = A.probabilities64(q[0, 0], k[0, 0], tau, False, np.arange(n))
    _, p2, _, _ = A.probabilities64(q2[0, 0], k2[0, 0], tau, False, np.arange(n))
    w = p1 * np.exp(c)[None, :]
    np.testing.assert_allclose(p2, w / w.sum(1, keepdims=True), atol=1e-15)


def _fd_grads(q, k, v, do, tau, causal, h=1e-5, fwd=None):
    fwd = fwd or oracle.attn_fwd64

    def f(qq, kk, vv):
        return float((fwd(qq, kk, vv, tau, causal)[0] * do).sum())

    out = []
    for which in range(3):
        args = [q.copy(), k.copy(), v.copy()]
        g = np.zeros_like(args[which])
        it = np.nditer(args[which], flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            a_p = [x.copy() for x in args]
            a_m = [x.copy() for x in args]
            a_p[which][idx] += h
            a_m[which][idx] -= h
            g[idx] = (f(*a_p) - f(*a_m)) / (2 * h)
        out.append(g)
    return out


@pytest.mark.parametrize("n,d,causal", [(1, 3, False), (5, 4, False), (7, 3, True), (9, 2, True), (6, 5, False)])
def test_backward_matches_finite_differences(n, d, causal):
    rng = np.random.default_rng(n * 31 + d)
    q, k, v, do = (rng.standard_normal((1, 2, n, d)) for _ in range(4))
    tau = 0.8
    dq, dk, dv, _ = oracle.attn_bwd64(q, k, v, do, tau, causal)
    fq, fk, fv = _fd_grads(q, k, v, do, tau, causal)
    for a, b in ((dq, fq), (dk, fk), (dv, fv)):
        assert np.abs(a - b).max() < 1e-8


def test_d_identity():
    rng = np.random.default_rng(3)
    q, k, v, do = (rng.standard_normal((2, 2, 40, 8)) for _ in range(4))
    for causal in (False, True):
        o, _ = oracle.attn_fwd64(q, k, v, 0.4, causal)
        _, _, _, dd = oracle.attn_bwd64(q, k, v, do, 0.4, causal)
        np.testing.assert_allclose(dd, (do * o).sum(-1), atol=1e-13, rtol=0)


# --------------------------------------------------------------------------
# sampled paths agree with the full definition
# --------------------------------------------------------------------------


@pytest.mark.parametrize("causal", [False, True])
def test_sampled_paths_match_full(causal):
    rng = np.random.default_rng(11)
    b_, h_, n, d = 2, 2, 70, 8
    q, k, v, do = (rng.standard_normal((b_, h_, n, d)) for _ in range(4))
    tau = 0.35
    o, lse = oracle.attn_fwd64(q, k, v, tau, causal)
    dq, dk, dv, dd = oracle.attn_bwd64(q, k, v, do, tau, causal)
    samples = np.array([[0, 0, 0], [1, 1, 69], [0, 1, 33], [1, 0, 5]])
    so, sl = oracle.attn_fwd64_rows(q, k, v, tau, causal, samples)
    sq, sd = oracle.attn_bwd64_query_rows(q, k, v, do, tau, causal, samples)
    for t, (b, h, i) in enumerate(samples):
        np.testing.assert_allclose(so[t], o[b, h, i], atol=1e-14)
        np.testing.assert_allclose(sl[t], lse[b, h, i], atol=1e-14)
        np.testing.assert_allclose(sq[t], dq[b, h, i], atol=1e-13)
        np.testing.assert_allclose(sd[t], dd[b, h, i], atol=1e-13)
    keys = np.array([0, 7, 69, 40])
    skk, svv = oracle.attn_bwd64_key_rows(q, k, v, do, tau, causal, 1, 0, keys)
    np.testing.assert_allclose(skk, dk[1, 0, keys], atol=1e-13)
    np.testing.assert_allclose(svv, dv[1, 0, keys], atol=1e-13)


# --------------------------------------------------------------------------
# planted mistakes: each slip below is caught by one of the pins above
# --------------------------------------------------------------------------


def _bwd_dropped_d(q, k, v, do, tau, causal):
    """Copy of the definition's backward with the −D term dropped from dS."""
    q, k, v, do = (np.asarray(t, float) for t in (q, k, v, do))
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    for b in range(q.shape[0]):
        for h in range(q.shape[1]):
            rows = np.arange(q.shape[2])
            _, p, _, _ = A.probabilities64(q[b, h], k[b, h], tau, causal, rows)
            dp = do[b, h] @ v[b, h].T
            ds = p * dp
            dv[b, h] = p.T @ do[b, h]
            dq[b, h] = tau * ds @ k[b, h]
            dk[b, h] = tau * ds.T @ q[b, h]
    return dq, dk, dv


def test_planted_dropped_d_term_fails_fd():
    rng = np.random.default_rng(5)
    q, k, v, do = (rng.standard_normal((1, 1, 5, 3)) for _ in range(4))
    bq, bk, _ = _bwd_dropped_d(q, k, v, do, 0.8, False)
    fq, fk, _ = _fd_grads(q, k, v, do, 0.8, False)
    assert np.abs(bq - fq).max() > 1e-3 and np.abs(bk - fk).max() > 1e-3


def test_planted_transposed_probabilities_fail_prefix_means():
    n, d = 6, 2
    q = _rand(1, 1, n, d)
    k = np.broadcast_to(_rand(1, 1, 1, d), (1, 1, n, d)).copy()
    v = _rand(1, 1, n, d)
    _, p, _, _ = A.probabilities64(q[0, 0], k[0, 0], 1.0, True, np.arange(n))
    wrong = p.T @ v[0, 0]
    prefix = np.cumsum(v[0, 0], axis=0) / np.arange(1, n + 1)[:, None]
    assert np.abs(wrong - prefix).max() > 1e-3


def test_planted_missing_rescale_fails_worked_example(golden):
    kv, rows = golden("online_softmax_worked_example.txt")
    x, blk = kv["x"], 3
    m, ell, trace = -math.inf, 0.0, []
    for s in range(0, len(x), blk):
        b = x[s:s + blk]
        m_new = max(m, max(b))
        ell = ell + sum(math.exp(t - m_new) for t in b)  # slip: old ℓ not rescaled
        m = m_new
        trace.append(ell)
    assert any(abs(a - r[2]) > 1e-3 for a, r in zip(trace, rows))


def test_planted_wrong_sign_fails_probability_rows():
    s = _rand(4, 7)
    m = s.max(1, keepdims=True)
    e = np.exp(m - s)  # slip: sign flipped
    p = e / e.sum(1, keepdims=True)
    _, p_ok, _, _ = A.probabilities64(s, np.eye(7), 1.0, False, np.arange(4))
    assert np.abs(p - p_ok).max() > 1e-2


def test_planted_missing_tau_in_dk_fails_fd():
    rng = np.random.default_rng(6)
    q, k, v, do = (rng.standard_normal((1, 1, 4, 3)) for _ in range(4))
    _, dk, _, _ = oracle.attn_bwd64(q, k, v, do, 0.5, False)
    _, fk, _ = _fd_grads(q, k, v, do, 0.5, False)
    assert np.abs(dk / 0.5 - fk).max() > 1e-3


# --------------------------------------------------------------------------
# grouped-query / multi-query attention
# --------------------------------------------------------------------------

from oracle import gqa as G  # noqa: E402


def test_gqa_group_of_one_is_plain_attention():
    rng = np.random.default_rng(21)
    q, k, v, do = (rng.standard_normal((2, 3, 11, 4)) for _ in range(4))
    for causal in (False, True):
        o1, l1 = G.attn_fwd64_gqa(q, k, v, 0.6, causal)
        o2, l2 = oracle.attn_fwd64(q, k, v, 0.6, causal)
        np.testing.assert_array_equal(o1, o2)
        np.testing.assert_array_equal(l1, l2)
        g1 = G.attn_bwd64_gqa(q, k, v, do, 0.6, causal)
        g2 = oracle.attn_bwd64(q, k, v, do, 0.6, causal)
        for a, b in zip(g1, g2):
            np.testing.assert_array_equal(a, b)


def test_gqa_heads_share_key_value_heads():
    # query heads 0,1 read key/value head 0; heads 2,3 read head 1 (g = 2)
    rng = np.random.default_rng(22)
    q = rng.standard_normal((1, 4, 9, 3))
    k, v = rng.standard_normal((1, 2, 9, 3)), rng.standard_normal((1, 2, 9, 3))
    o, _ = G.attn_fwd64_gqa(q, k, v, 0.5, True)
    for h in range(4):
        kv = G.kv_head_of(h, 4, 2)
        assert kv == h // 2
        oh, _ = oracle.attn_fwd64(q[:, h:h + 1], k[:, kv:kv + 1], v[:, kv:kv + 1], 0.5, True)
        np.testing.assert_allclose(o[:, h], oh[:, 0], atol=1e-15)
    with pytest.raises(ValueError):
        G.kv_head_of(0, 4, 3)


@pytest.mark.parametrize("h,h_kv,causal", [(4, 2, False), (3, 1, True)])
def test_gqa_backward_matches_finite_differences(h, h_kv, causal):
    rng = np.random.default_rng(23 + h)
    n, d = 5, 3
    q, do = rng.standard_normal((1, h, n, d)), rng.standard_normal((1, h, n, d))
    k, v = rng.standard_normal((1, h_kv, n, d)), rng.standard_normal((1, h_kv, n, d))
    dq, dk, dv, _ = G.attn_bwd64_gqa(q, k, v, do, 0.7, causal)
    fq, fk, fv = _fd_grads(q, k, v, do, 0.7, causal, fwd=G.attn_fwd64_gqa)
    for a, b in ((dq, fq), (dk, fk), (dv, fv)):
        assert np.abs(a - b).max() < 1e-8


def test_planted_gqa_backward_without_group_sum_fails_fd():
    rng = np.random.default_rng(29)
    q, do = rng.standard_normal((1, 2, 4, 3)), rng.standard_normal((1, 2, 4, 3))
    k, v = rng.standard_normal((1, 1, 4, 3)), rng.standard_normal((1, 1, 4, 3))
    _, dk_e, _, _ = oracle.attn_bwd64(q, G.expand_kv(k, 2), G.expand_kv(v, 2), do, 0.7, False)
    wrong = dk_e[:, :1]  # slip: only the first query head's contribution
    _, fk, _ = _fd_grads(q, k, v, do, 0.7, False, fwd=G.attn_fwd64_gqa)
    assert np.abs(wrong - fk).max() > 1e-3


# --------------------------------------------------------------------------
# decoding over a long cache, split into pieces and merged (Flash-Decoding)
# --------------------------------------------------------------------------

from oracle import decode as DEC  # noqa: E402


@pytest.mark.parametrize("splits", [1, 2, 3, 7, 40])
def test_split_kv_merge_equals_whole_cache(splits):
    rng = np.random.default_rng(31 + splits)
    q = rng.standard_normal((2, 4, 3, 8))
    k, v = rng.standard_normal((2, 2, 37, 8)) * 2, rng.standard_normal((2, 2, 37, 8))
    o_ref, l_ref = DEC.decode_fwd64(q, k, v, 0.4)
    o, lse = DEC.merge_splits64(DEC.split_kv_states64(q, k, v, 0.4, splits))
    np.testing.assert_allclose(o, o_ref, atol=1e-14)
    np.testing.assert_allclose(lse, l_ref, atol=1e-13)


def test_decode_is_attention_over_the_whole_cache():
    # one query row equal to the last row of a square problem: same output as that row
    rng = np.random.default_rng(41)
    q, k, v = (rng.standard_normal((1, 2, 20, 6)) for _ in range(3))
    o_full, l_full = oracle.attn_fwd64(q, k, v, 0.5, False)
    o, lse = DEC.decode_fwd64(q[:, :, -1:], k, v, 0.5)
    np.testing.assert_allclose(o[:, :, 0], o_full[:, :, -1], atol=1e-15)
    np.testing.assert_allclose(lse[:, :, 0], l_full[:, :, -1], atol=1e-15)
    # a single cached key: O = V, L = τ q·k
    o1, l1 = DEC.decode_fwd64(q[:, :, :3], k[:, :, :1], v[:, :, :1], 0.5)
    np.testing.assert_array_equal(o1, np.broadcast_to(v[:, :, :1], o1.shape))
    np.testing.assert_allclose(l1, 0.5 * (q[:, :, :3] @ k[:, :, 0, :, None])[..., 0], atol=1e-15)


def test_split_bounds_cover_the_cache():
    for nk, s in [(1, 1), (10, 3), (4097, 16), (5, 8)]:
        b = DEC.split_bounds(nk, s)
        assert b[0][0] == 0 and b[-1][1] == nk and len(b) == s
        assert all(b[i][1] == b[i + 1][0] for i in range(s - 1))


def test_planted_merge_without_rescale_fails():
    rng = np.random.default_rng(43)
    q = rng.standard_normal((1, 1, 1, 4))
    k, v = rng.standard_normal((1, 1, 10, 4)) * 3, rng.standard_normal((1, 1, 10, 4))
    (m1, l1, o1), (m2, l2, o2) = DEC.split_kv_states64(q, k, v, 1.0, 2)
    wrong = (l1 * o1 + l2 * o2) / (l1 + l2)  # slip: partial states not brought to a common maximum
    o_ref, _ = DEC.decode_fwd64(q, k, v, 1.0)
    assert np.abs(wrong - o_ref).max() > 1e-3


# --------------------------------------------------------------------------
# FP8 (E4M3) block quantisation and the attention it feeds
# --------------------------------------------------------------------------

from oracle import fp8 as F8  # noqa: E402


def test_e4m3_value_set_from_the_format():
    v = F8.e4m3_values()
    assert len(v) == 127  # zero, 7 subnormals, 15 binades x 8 mantissas minus the NaN code
    assert v[0] == 0 and v[1] == 2.0 ** -9 and v[7] == 7 * 2.0 ** -9 and v[8] == 2.0 ** -6
    assert v[-1] == 448.0 and v[-2] == 416.0
    assert np.all(np.diff(v) > 0)


def test_e4m3_round_fixes_values_and_takes_ties_to_even():
    v = F8.e4m3_values()
    np.testing.assert_array_equal(F8.e4m3_round(v), v)
    np.testing.assert_array_equal(F8.e4m3_round(-v[1:]), -v[1:])
    mid = (v[:-1] + v[1:]) / 2
    # codes ascend with the value and the mantissa is the code's low 3 bits: the even-index
    # neighbour has the even mantissa
    want = np.where(np.arange(len(mid)) % 2 == 0, v[:-1], v[1:])
    np.testing.assert_array_equal(F8.e4m3_round(mid), want)
    # just off the midpoints: the nearer neighbour
    np.testing.assert_array_equal(F8.e4m3_round(mid * (1 - 1e-9)), v[:-1])
    np.testing.assert_array_equal(F8.e4m3_round(mid * (1 + 1e-9)), v[1:])
    # saturation (satfinite): everything above 448 is 448
    np.testing.assert_array_equal(F8.e4m3_round([449.0, 470.0, 1e6, -1e6]), [448.0, 448.0, 448.0, -448.0])
    assert F8.e4m3_round(2.0 ** -11) == 0.0 and F8.e4m3_round(3 * 2.0 ** -11) == 2.0 ** -9


def test_e4m3_round_matches_the_torch_float8_conversion():
    torch = pytest.importorskip("torch")
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("no float8 dtype in this torch")
    rng = np.random.default_rng(71)
    x = np.concatenate([rng.standard_normal(20000) * s for s in (1e-3, 0.05, 1.0, 30.0, 150.0)])
    x = x[np.abs(x) <= 448.0]
    ref = torch.from_numpy(x.astype(np.float32)).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    np.testing.assert_array_equal(F8.e4m3_round(x.astype(np.float32)), ref)


def test_block_quantisation_scales_each_block_to_the_format_range():
    rng = np.random.default_rng(72)
    x = rng.standard_normal((2, 3, 300, 16)) * rng.uniform(0.01, 100, size=(2, 3, 1, 1))
    codes, scales = F8.quantize_blocks(x)
    assert scales.shape == (2, 3, 3) and scales.dtype == np.float32
    for b in range(3):
        blk = codes[:, :, b * 128:(b + 1) * 128]
        np.testing.assert_array_equal(np.abs(blk).max(axis=(-2, -1)), 448.0)  # each block's amax maps to 448
        np.testing.assert_array_equal(F8.e4m3_round(blk), blk)  # codes are E4M3 values
        np.testing.assert_allclose(scales[..., b], np.abs(x[:, :, b * 128:(b + 1) * 128]).max(axis=(-2, -1)) / 448,
                                   rtol=1e-7)
    deq = F8.dequantize_blocks(codes, scales)
    # E4M3 keeps 3 mantissa bits: relative error <= 2^-4 above the subnormal range
    big = np.abs(x) >= np.repeat(scales, 128, axis=-1)[..., :300, None] * 2.0 ** -6
    assert np.all(np.abs(deq - x)[big] <= 2.0 ** -4 * np.abs(x)[big] * (1 + 1e-6))
    # zero block: scale 1, codes 0
    z_codes, z_scales = F8.quantize_blocks(np.zeros((1, 1, 5, 8)))
    assert z_scales[0, 0, 0] == 1.0 and not z_codes.any()


def test_block_quantisation_beats_one_scale_per_tensor():
    # blocks of very different magnitude (the case block quantisation is for): one scale for
    # the whole tensor pushes the small blocks into the subnormal range
    rng = np.random.default_rng(73)
    mags = np.array([1e-3, 1.0, 50.0, 1e-2])
    x = rng.standard_normal((1, 1, 512, 64)) * np.repeat(mags, 128)[None, None, :, None]
    codes, scales = F8.quantize_blocks(x)
    err_block = np.linalg.norm(F8.dequantize_blocks(codes, scales) - x) / np.linalg.norm(x)
    c1, s1 = F8.quantize_blocks(x, block=512)  # one block = one scale for the tensor
    small = x[..., :128, :]

    def rel(deq):
        return np.linalg.norm(deq[..., :128, :] - small) / np.linalg.norm(small)

    # E4M3 rounding keeps every normal value within 2^-4 (RMS about 2^-3 / sqrt(12) = 0.036)
    assert err_block < 0.036
    assert rel(F8.dequantize_blocks(codes, scales)) < 0.036
    assert rel(F8.dequantize_blocks(c1, s1, block=512)) > 5 * rel(F8.dequantize_blocks(codes, scales))


def test_fp8_attention_is_attention_on_the_dequantised_inputs():
    rng = np.random.default_rng(74)
    # inputs that are E4M3 values with a block maximum of 448: scale 1, dequantisation exact
    v = F8.e4m3_values()
    q, k, vv = (rng.choice(np.concatenate([v, -v]), size=(1, 2, 130, 16)) for _ in range(3))
    for t in (q, k, vv):
        t[..., 0, 0] = 448.0
        t[..., 128, 0] = 448.0
    qc, qs = F8.quantize_blocks(q)
    kc, ks = F8.quantize_blocks(k)
    vc, vs = F8.quantize_blocks(vv)
    assert np.all(qs == 1) and np.array_equal(qc, q)
    o, lse = F8.attn_fwd64_fp8(qc, qs, kc, ks, vc, vs, 0.01, True)
    o_ref, l_ref = oracle.attn_fwd64(q, k, vv, 0.01, True)
    np.testing.assert_array_equal(o, o_ref)
    np.testing.assert_array_equal(lse, l_ref)


def test_planted_truncating_e4m3_fails():
    v = F8.e4m3_values()
    mid = (v[:-1] + v[1:]) / 2

    def truncating(x):  # slip: rounds toward zero instead of to nearest
        a = np.abs(x)
        _, fe = np.frexp(np.where(a > 0, a, 1.0))
        ulp = 2.0 ** (np.maximum(fe - 1, -6) - 3)
        return np.floor(a / ulp) * ulp

    want = np.where(np.arange(len(mid)) % 2 == 0, v[:-1], v[1:])
    assert not np.array_equal(truncating(mid), want)


# --------------------------------------------------------------------------
# block-sparse and sliding-window masks (Lecture 8 §5.7, Proposition 4)
# --------------------------------------------------------------------------

from oracle import masks as MK  # noqa: E402


def _qkv(seed, b=1, h=2, n=40, d=6):
    rng = np.random.default_rng(seed)
    return tuple(rng.standard_normal((b, h, n, d)) for _ in range(3))


def test_mask_special_cases_reduce_to_the_known_masks():
    n, blk = 40, 8
    nb = n // blk
    assert MK.visible_mask(n, block_mask=np.ones((nb, nb)), block=blk).all()
    np.testing.assert_array_equal(MK.visible_mask(n, True, block_mask=np.tril(np.ones((nb, nb))), block=blk),
                                  MK.visible_mask(n, True))
    np.testing.assert_array_equal(MK.visible_mask(n, True, window=n), MK.visible_mask(n, True))
    vis = MK.visible_mask(n, True, window=5)
    np.testing.assert_array_equal(vis.sum(axis=1), np.minimum(np.arange(n) + 1, 5))
    vis2 = MK.visible_mask(n, False, window=5)
    np.testing.assert_array_equal(vis2.sum(axis=1), [min(i, 4) + min(n - 1 - i, 4) + 1 for i in range(n)])


def test_masked_definition_agrees_with_the_standard_one():
    q, k, v = _qkv(81)
    n = q.shape[2]
    for causal in (False, True):
        o, lse = MK.attn_fwd64_masked(q, k, v, 0.4, MK.visible_mask(n, causal))
        o_ref, l_ref = oracle.attn_fwd64(q, k, v, 0.4, causal)
        np.testing.assert_allclose(o, o_ref, atol=1e-14)
        np.testing.assert_allclose(lse, l_ref, atol=1e-14)


def test_window_of_one_and_local_windows_in_closed_form():
    q, k, v = _qkv(82)
    n = q.shape[2]
    o, lse = MK.attn_fwd64_masked(q, k, v, 0.7, MK.visible_mask(n, True, window=1))
    np.testing.assert_allclose(o, v, atol=1e-15)
    np.testing.assert_allclose(lse, 0.7 * np.einsum("bhnd,bhnd->bhn", q, k), atol=1e-14)
    # a causal window of w: row i is ordinary attention over keys i-w+1 .. i
    w = 6
    o, lse = MK.attn_fwd64_masked(q, k, v, 0.7, MK.visible_mask(n, True, window=w))
    for i in (0, 3, 5, 6, 17, n - 1):
        lo = max(0, i - w + 1)
        s = 0.7 * k[0, 1, lo:i + 1] @ q[0, 1, i]
        p = np.exp(s - s.max())
        np.testing.assert_allclose(o[0, 1, i], p @ v[0, 1, lo:i + 1] / p.sum(), atol=1e-14)
        np.testing.assert_allclose(lse[0, 1, i], s.max() + np.log(p.sum()), atol=1e-14)


def test_block_diagonal_mask_is_independent_attention_per_block():
    q, k, v = _qkv(83, n=48)
    blk = 16
    bm = np.eye(3)
    o, lse = MK.attn_fwd64_masked(q, k, v, 0.3, MK.visible_mask(48, block_mask=bm, block=blk))
    for c in range(3):
        sl = slice(c * blk, (c + 1) * blk)
        o_ref, l_ref = oracle.attn_fwd64(q[:, :, sl], k[:, :, sl], v[:, :, sl], 0.3, False)
        np.testing.assert_allclose(o[:, :, sl], o_ref, atol=1e-14)
        np.testing.assert_allclose(lse[:, :, sl], l_ref, atol=1e-14)


def test_rows_with_no_visible_key():
    q, k, v = _qkv(84, n=32)
    bm = np.ones((4, 4))
    bm[2, :] = 0  # query block 2 sees nothing
    vis = MK.visible_mask(32, block_mask=bm, block=8)
    o, lse = MK.attn_fwd64_masked(q, k, v, 0.5, vis)
    assert np.all(o[:, :, 16:24] == 0) and np.all(lse[:, :, 16:24] == -np.inf)
    rng = np.random.default_rng(85)
    do = rng.standard_normal(q.shape)
    dq, dk, dv = MK.attn_bwd64_masked(q, k, v, do, 0.5, vis)
    assert np.all(dq[:, :, 16:24] == 0)
    # those rows' dO reaches no key: changing it leaves dK, dV unchanged
    do2 = do.copy()
    do2[:, :, 16:24] += 3.0
    _, dk2, dv2 = MK.attn_bwd64_masked(q, k, v, do2, 0.5, vis)
    np.testing.assert_array_equal(dk, dk2)
    np.testing.assert_array_equal(dv, dv2)


def test_block_sparse_tiled_forward_equals_definition_and_visits_nonzero_blocks():
    rng = np.random.default_rng(86)
    n, blk = 70, 16
    nb = (n + blk - 1) // blk
    q, k, v = (rng.standard_normal((n, 8)) for _ in range(3))
    for causal, window, dens in [(False, 0, 0.5), (True, 0, 0.6), (True, 20, 1.0), (False, 9, 0.7), (True, 0, 1.0)]:
        bm = (rng.random((nb, nb)) < dens).astype(np.uint8)
        bm[:, 0] = 1  # every row sees at least its first block unless the window removes it
        vis = MK.visible_mask(n, causal, window, bm, blk)
        o, lse, visited = MK.tiled_fwd_block_sparse(q, k, v, 0.45, vis, blk)
        o_ref, l_ref = MK.attn_fwd64_masked(q[None, None], k[None, None], v[None, None], 0.45, vis)
        np.testing.assert_allclose(o, o_ref[0, 0], atol=1e-13)
        np.testing.assert_allclose(lse, l_ref[0, 0], atol=1e-13)
        assert visited == MK.blocks_visited(n, causal, window, bm, blk).sum()
    # the causal example of the page: 136 of 16 x 16 blocks
    assert MK.blocks_visited(16 * 128, True).sum() == 136


def test_masked_backward_against_finite_differences():
    rng = np.random.default_rng(87)
    n, d, blk = 10, 3, 4
    q, k, v, do = (rng.standard_normal((1, 1, n, d)) for _ in range(4))
    bm = np.array([[1, 0, 1], [1, 1, 0], [0, 1, 1]])
    vis = MK.visible_mask(n, True, 4, bm, blk)
    dq, dk, dv = MK.attn_bwd64_masked(q, k, v, do, 0.6, vis)

    def f(q_, k_, v_):
        return (MK.attn_fwd64_masked(q_, k_, v_, 0.6, vis)[0] * do).sum()

    h = 1e-6
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            args = {"q": q, "k": k, "v": v}
            args[name] = xp
            fp = f(args["q"], args["k"], args["v"])
            args[name] = xm
            fm = f(args["q"], args["k"], args["v"])
            num[idx] = (fp - fm) / (2 * h)
        np.testing.assert_allclose(g, num, atol=1e-8, rtol=1e-6)


def test_planted_window_off_by_one_fails():
    q, k, v = _qkv(88)
    n = q.shape[2]
    wrong = np.abs(np.arange(n)[:, None] - np.arange(n)[None, :]) <= 1  # slip: <= w instead of < w
    wrong &= np.arange(n)[None, :] <= np.arange(n)[:, None]
    o, _ = MK.attn_fwd64_masked(q, k, v, 0.7, wrong)
    assert np.abs(o - v).max() > 1e-3  # the window-of-one closed form O = V catches it


def test_masked_sampled_rows_equal_the_full_definition():
    q, k, v = _qkv(89, b=2, h=3, n=50)
    rng = np.random.default_rng(90)
    bm = (rng.random((3, 4, 4)) < 0.6).astype(np.uint8)
    for causal, window in [(True, 7), (False, 12), (True, 0)]:
        vis = MK.visible_mask(50, causal, window, bm, 16)
        o, lse = MK.attn_fwd64_masked(q, k, v, 0.5, vis)
        samples = [(0, 0, 0), (1, 2, 49), (0, 1, 17), (1, 0, 33)]
        o_r, l_r = MK.attn_fwd64_masked_rows(q, k, v, 0.5, samples, causal, window, bm, 16)
        for t, (b, h, i) in enumerate(samples):
            np.testing.assert_allclose(o_r[t], o[b, h, i], atol=1e-15)
            np.testing.assert_allclose(l_r[t], lse[b, h, i], atol=1e-15)
