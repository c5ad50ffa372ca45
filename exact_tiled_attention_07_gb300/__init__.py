"""Exact tiled attention (forward + recomputing backward) for NVIDIA GB300, sm_103a.

The computation lives in ``libfa_gb300.so`` (C ABI: ``include/fa.h``): TMA-fed
tcgen05 kernels for bf16/fp16 and CUDA-core kernels for fp32.  ``binding``
marshals torch tensors into those calls; ``inputs`` draws the seeded synthetic
workloads.  Build with ``python -m exact_tiled_attention_07_gb300.build``.
"""

from . import inputs  # noqa: F401

__all__ = ["inputs", "binding"]


def __getattr__(name):
    # the binding imports torch; load it on first use
    if name == "binding":
        import importlib

        mod = importlib.import_module(".binding", __name__)
        globals()["binding"] = mod
        return mod
    raise AttributeError(name)
