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
# L: S = Q8 K8^T is accumulated by the tensor core, whose sum of 8-bit products is not an
# IEEE fp32 sum; the dot-product error bound |dS| <= k u sum|q_k k_k| with the unit roundoff u
# of that accumulation gives an L error proportional to the row's largest |S|.  Read here as
# |dL| <= 1e-3 + 2^-11 max_j |S_ij| (u about 2^-14, the measured relative error of L at large
# scores being about 2^-13).
TOL_FP8_L_OF_SMAX = 2.0 ** -11

