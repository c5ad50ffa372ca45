"""Shared test helpers: moving seeded inputs to the device and comparison metrics."""

import numpy as np

TORCH_DT = {}


def torch_dtype(name):
    import torch

    return {"fp32": torch.float32, "fp16": torch.float16, "bf16": torch.bfloat16}[name]


def to_device(stored, dtype, device="cuda"):
    """Storage array from exact_tiled_attention_07_gb300.inputs -> torch tensor on the device."""
    import torch

    if dtype == "bf16":
        t = torch.from_numpy(np.ascontiguousarray(stored).view(np.int16)).view(torch.bfloat16)
    else:
        t = torch.from_numpy(np.ascontiguousarray(stored))
    return t.to(device)


def to_f64(t):
    """torch tensor (any float dtype, any device) -> float64 numpy."""
    import torch

    return t.detach().to("cpu", torch.float64).numpy()


def max_abs(x, y):
    return float(np.max(np.abs(np.asarray(x, np.float64) - np.asarray(y, np.float64)))) if np.size(x) else 0.0


def rel_rms(x, y):
    x = np.asarray(x, np.float64)
    y = np.asarray(y, np.float64)
    den = np.sqrt(np.mean(y * y))
    return float(np.sqrt(np.mean((x - y) ** 2)) / den) if den > 0 else float(np.sqrt(np.mean((x - y) ** 2)))


# Tolerances (the fp64 oracle is the reference):
#   16-bit O: max-abs <= 1e-2 and rel-RMS <= 5e-3; dQ/dK/dV: rel-RMS <= 1e-2; L: max-abs <= 1e-3
#   fp32 path: max-abs <= 1e-5 on O, L, dQ, dK, dV
TOL_O_MAXABS = 1e-2
TOL_O_RELRMS = 5e-3
TOL_GRAD_RELRMS = 1e-2
TOL_L_MAXABS = 1e-3
TOL_FP32 = 1e-5

# FP8 forward against attention on the dequantised inputs.  The kernel rounds P (scaled into
# (0, 2^8]) to E4M3 before the P V product: each probability carries a relative error of at
# most 2^-4 (3 mantissa bits, round to nearest), RMS 2^-3 / sqrt(12) ~ 0.036 for a uniformly
# spread rounding error, so O's relative RMS error is about 0.036 and |error| of an element
# is at most 2^-4 max|V| (the weights sum to one).  L does not involve the rounded P.
TOL_FP8_O_RELRMS = 0.05
TOL_FP8_O_MAXABS_OF_VMAX = 2.0 ** -4
# L: S = Q8 K8^T comes from the tensor core's sums of 8-bit products, whose internal precision
# the PTX ISA does not state.  Model, an assumption: every product of two E4M3 values is exact
# (at most 8 significant bits); each MMA instruction adds its K = 32 products and rounds that
# group sum G once, keeping at least 13 significant bits and possibly truncating (error below
# 2^-12 |G|); the group sums then enter the fp32 accumulator (d / 32 additions, 2^-24 each).
# Summed over the groups, |dS_ij| <= u tau sum_k |q_ik k_jk| (dequantised values) with
# u = 2^-12 + (d / 32) 2^-24, and since dL_i / dS_ij = P_ij sums to one over j,
# |dL_i| <= max_j |dS_ij|.  The check on exactly representable inputs (codes whose group sums
# need 13 significant bits) tests the 13-bit part of the model: there L meets the plain 1e-3.
TOL_FP8_ACC_U = 2.0 ** -12 + 4 * 2.0 ** -24



def key_side_reference(job):
    """One head's exact key-side gradients from the fp64 oracle (a process-pool worker).

    job = (q, k, v, do, scale, causal, keys) with q, k, v, do the head's [1, 1, N, d] fp64
    inputs.  dK_j, dV_j need every row's L_i and D_i (column j of P involves each row's
    normalisation), so the head's statistics are computed first.  Returns (dK [keys, d],
    dV [keys, d], L [N]).
    """
    import oracle

    q, k, v, do, scale, causal, keys = job
    stats = oracle.attn_stats64(q, k, v, do, scale, causal, 0, 0)
    dk, dv = oracle.attn_bwd64_key_rows(q, k, v, do, scale, causal, 0, 0, keys, stats=stats)
    return dk, dv, stats[0]


def oracle_pool_map(fn, jobs, threads_per_worker=2):
    """fn over jobs in a pool of spawned processes (never forked: the parent holds a CUDA
    context), each with its BLAS limited to a few threads so the workers share the cores."""
    import multiprocessing as mp
    import os

    names = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")
    saved = {n: os.environ.get(n) for n in names}
    workers = max(1, min(len(jobs), (os.cpu_count() or 2) // threads_per_worker))
    try:
        for n in names:
            os.environ[n] = str(threads_per_worker)
        with mp.get_context("spawn").Pool(workers) as pool:
            return pool.map(fn, jobs)
    finally:
        for n, v in saved.items():
            if v is None:
                os.environ.pop(n, None)
            else:
                os.environ[n] = v
