"""The process pool the full-size GPU tests use for the oracle's key-side gradients (CPU only):
spawned workers return what the oracle returns in this process (to the rounding of a BLAS
that may split its sums differently with fewer threads)."""

import numpy as np

import oracle
from helpers import key_side_reference, oracle_pool_map


def test_pool_workers_match_the_oracle_called_directly():
    rng = np.random.default_rng(7)
    jobs = []
    for h in range(3):
        q, k, v, do = (rng.standard_normal((1, 1, 200, 16)) for _ in range(4))
        jobs.append((q, k, v, do, 0.25, bool(h % 2), np.array([0, 17, 127, 128, 199])))
    got = oracle_pool_map(key_side_reference, jobs)
    for job, (dk, dv, lse) in zip(jobs, got):
        q, k, v, do, scale, causal, keys = job
        stats = oracle.attn_stats64(q, k, v, do, scale, causal, 0, 0)
        dk_ref, dv_ref = oracle.attn_bwd64_key_rows(q, k, v, do, scale, causal, 0, 0, keys, stats=stats)
        np.testing.assert_allclose(dk, dk_ref, rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(dv, dv_ref, rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(lse, stats[0], rtol=1e-12, atol=1e-13)
        # and the key rows agree with the whole backward of the definition
        dq_full, dk_full, dv_full, _ = oracle.attn_bwd64(q, k, v, do, scale, causal)
        np.testing.assert_allclose(dk, dk_full[0, 0, keys], rtol=0, atol=1e-12)
        np.testing.assert_allclose(dv, dv_full[0, 0, keys], rtol=0, atol=1e-12)
