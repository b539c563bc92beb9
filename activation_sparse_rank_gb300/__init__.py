"""Predictor-gated, neuron-aware sparse FFN for one NVIDIA GB300 (sm_103a).

Python face of libpi (``include/pi.h``): ctypes marshalling of torch device
tensors and streams onto the C ABI.  Every step of the computation runs in
the CUDA library; there is no fallback.  Importing this package raises if
libpi.so has not been built (``python activation_sparse_rank_gb300/_build.py``).
"""
from .binding import (  # noqa: F401
    PI_ACT_REGLU,
    PI_ACT_SWIGLU,
    PI_ACT_RELU,
    PI_MAX_BATCH,
    PI_STACK_LAYERS_PER_LAUNCH,
    Layer,
    PiError,
    hot_first_perm,
    lib,
    lib_path,
    profile_activations,
    stack_forward,
    stack_forward_host,
)

__all__ = [
    "Layer",
    "PiError",
    "PI_ACT_RELU",
    "PI_ACT_REGLU",
    "PI_ACT_SWIGLU",
    "PI_MAX_BATCH",
    "PI_STACK_LAYERS_PER_LAUNCH",
    "hot_first_perm",
    "lib",
    "lib_path",
    "profile_activations",
    "stack_forward",
    "stack_forward_host",
]
