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
