"""The five synthetic FFN workloads, by shape.

Each one stands in for a model family the PowerInfer paper evaluates
("PowerInfer: Fast LLM Serving with a Consumer-grade GPU", egguo-blog reading
report, section 2.2 "Data source": OPT 7B-175B and Falcon-40B with ReLU,
LLaMA2-70B with ReGLU) and for the decode setting of section 2.2 (inputs of
8-128 tokens).  The firing-rate skew (Zipf exponent) and the mean sparsity
stand in for the power-law activation locality of section 3.1, Finding 1.
The SwiGLU shape follows section 4.4, limitation 1 (SwiGLU models keep about
half of their neurons).
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Tuple


@dataclass(frozen=True)
class LayerSpec:
    d: int                 # model width
    ffn: int               # number of FFN neurons
    rank: int              # predictor hidden width r
    act: str = "relu"      # "relu", "reglu" or "swiglu"
    alpha: float = 1.0     # Zipf exponent of the per-neuron firing rates
    mean_f: float = 0.10   # mean firing rate (1 - sparsity)
    f_cap: float = 0.9     # cap on any single neuron's firing rate
    w_std: float = 0.02    # std of W_up / W_gate / W_down entries
    wp_std: float = 0.05   # std of W_p1 / W_p2 entries
    predictor_bias: str = "calibrated"   # "calibrated" or "none"


@dataclass(frozen=True)
class StackConfig:
    name: str
    layer: LayerSpec
    layers: int
    tokens: int
    batches: Tuple[int, ...] = (1,)
    prompt: int = 0              # tokens processed together in a prompt pass
    profile_tokens: int = 0      # tokens of the hot-first profiling run (0: identity order)
    seed: int = 1000
    description: str = field(default="", compare=False)


CONFIGS = (
    StackConfig(
        name="opt_layer_d1024",
        layer=LayerSpec(d=1024, ffn=4096, rank=64, alpha=1.0, mean_f=0.10),
        layers=1, tokens=64, seed=1001,
        description="single OPT-style ReLU FFN layer, d=1024, ffn=4096, r=64, batch 1, 64 tokens",
    ),
    StackConfig(
        name="opt7b_stack",
        layer=LayerSpec(d=4096, ffn=16384, rank=256, alpha=1.0, mean_f=0.10),
        layers=32, tokens=256, profile_tokens=10000, seed=1002,
        description="OPT-7B-shaped ReLU FFN stack, d=4096, ffn=16384, 32 layers, r=256, "
                    "batch 1, 256 decode tokens, hot-first order from a 10k-token profile",
    ),
    StackConfig(
        name="llama2_70b_reglu",
        layer=LayerSpec(d=8192, ffn=28672, rank=512, act="reglu", alpha=0.8, mean_f=0.15),
        layers=16, tokens=256, seed=1003,
        description="LLaMA2-70B ReGLU-shaped FFN, d=8192, ffn=28672, 16 layers, r=512, batch 1",
    ),
    StackConfig(
        name="llama2_70b_swiglu",
        layer=LayerSpec(d=8192, ffn=28672, rank=512, act="swiglu", alpha=0.5, mean_f=0.5),
        layers=16, tokens=256, seed=1006,
        description="LLaMA2-70B SwiGLU-shaped FFN, d=8192, ffn=28672, 16 layers, r=512, batch 1, "
                    "about 50% of the neurons kept by the predictor",
    ),
    StackConfig(
        name="falcon40b_stack",
        layer=LayerSpec(d=8192, ffn=32768, rank=384, alpha=1.1, mean_f=0.08),
        layers=60, tokens=128, batches=(1, 2, 4, 8, 16, 32), seed=1004,
        description="Falcon-40B-shaped ReLU FFN, d=8192, ffn=32768, 60 layers, r=384, "
                    "batch sweep 1..32 (union active set)",
    ),
    StackConfig(
        name="opt175b_stack",
        layer=LayerSpec(d=12288, ffn=49152, rank=1024, alpha=1.0, mean_f=0.10),
        layers=8, tokens=64, batches=(1, 8, 32), prompt=128, seed=1005,
        description="OPT-175B-shaped ReLU FFN, d=12288, ffn=49152, 8 layers, r=1024, "
                    "batch 1/8/32 and a 128-token prompt pass",
    ),
)


def config_by_name(name: str) -> StackConfig:
    for c in CONFIGS:
        if c.name == name:
            return c
    raise KeyError(name)
