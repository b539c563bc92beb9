"""Seeded synthetic inputs for the predictor-gated sparse FFN.

This package only draws random numbers and builds weights of the shapes and
statistics the five workloads call for.  It holds none of the method's own
arithmetic (no predictor forward, no FFN, no active-set selection), so that
both the CPU oracle and the CUDA path can consume what it produces.
"""
from .configs import CONFIGS, LayerSpec, StackConfig, config_by_name
from .gen import (
    firing_rates,
    make_layer,
    make_tokens,
    make_exact_layer,
    make_exact_tokens,
    sub_seed,
)

__all__ = [
    "CONFIGS",
    "LayerSpec",
    "StackConfig",
    "config_by_name",
    "firing_rates",
    "make_layer",
    "make_tokens",
    "make_exact_layer",
    "make_exact_tokens",
    "sub_seed",
]
