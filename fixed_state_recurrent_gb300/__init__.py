"""Normalized causal linear attention (ELU+1) and the delta-rule memory on GB300.

The compute lives in ``libla.so`` (CUDA for sm_103a, C ABI declared in
``include/la.h``).  This package is a thin binding: ``prefill``,
``decode_step`` and ``delta_prefill`` marshal torch CUDA tensors to the C
entry points of the same names and launch on the current torch stream.  There
is no CPU fallback: calling them without the built library raises.
"""
from .inputs import WORKLOADS, Workload  # noqa: F401

__all__ = [
    "prefill", "decode_step", "delta_prefill", "prefill_workspace_bytes",
    "state_bytes", "read_device_status", "LAError", "WORKLOADS", "Workload",
]


def __getattr__(name):
    # The binding (and libla.so) is loaded on first use so that importing the
    # package for its input generators works on machines without a GPU.
    if name in ("prefill", "decode_step", "delta_prefill",
                "prefill_workspace_bytes", "state_bytes",
                "read_device_status", "LAError", "lib"):
        from . import api
        return getattr(api, name)
    raise AttributeError(name)
