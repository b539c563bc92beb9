"""CPU oracle for the predictor-gated sparse FFN (test infrastructure only).

This package is the plain, slow, float64 statement of what the GPU path
computes.  It exists to check the CUDA library: only the test-suite, the
smoke check and the benchmark's CPU-baseline leg may import it; the product
path never calls it and shares no code with it.

Source of the method: "PowerInfer: Fast Large Language Model Serving with a
Consumer-grade GPU" (egguo-blog reading report), section 2.3
"Operationalization & Measurement": the adaptive predictor (core module 3),
the neuron-aware sparse operators (core module 4), the definition of ReLU
sparsity as the fraction of exactly-zero activations, hot/cold neurons by
activation frequency and the neuron impact v_i = f_i; section 4.4
(batching: the active set grows as batch grows).

Parity status per function (pins live in tests/test_oracle_*.py):
  predictor_hidden / predictor_logits / predicted_mask   pinned
  active_union                                            pinned
  logit_error_bound / preact_error_bound                  pinned
  ffn_activations / ffn_output / sparse_ffn / dense_ffn   pinned
  profile_counts / hot_first_order / permute_layer        pinned
Predictor *accuracy* against true activations is parity unpinned: it needs
trained weights, which this build does not have.
"""
from .ffn import (
    OracleLayer,
    active_union,
    dense_ffn,
    exact_mask,
    ffn_activations,
    ffn_output,
    hot_first_order,
    logit_error_bound,
    permute_layer,
    preact_error_bound,
    predicted_forward,
    predicted_mask,
    predictor_hidden,
    predictor_logits,
    profile_counts,
    sparse_ffn,
)

__all__ = [
    "OracleLayer",
    "active_union",
    "dense_ffn",
    "exact_mask",
    "ffn_activations",
    "ffn_output",
    "hot_first_order",
    "logit_error_bound",
    "permute_layer",
    "preact_error_bound",
    "predicted_forward",
    "predicted_mask",
    "predictor_hidden",
    "predictor_logits",
    "profile_counts",
    "sparse_ffn",
]
