"""Seeded generators for FFN layers, predictor weights and decode tokens.

Construction (one layer, ``LayerSpec`` sizes):

* ``W_up``, ``W_gate`` ([ffn, d]) and ``W_down`` ([d, ffn]) are N(0, w_std^2),
  rounded to fp16.  ``W_p1`` ([r, d]) and ``W_p2`` ([ffn, r]) are
  N(0, wp_std^2), rounded to fp16.  Tokens are x ~ N(0, I), rounded to fp16.
* Firing rates follow the power law of "PowerInfer" (egguo-blog report,
  section 3.1 Finding 1 and Figure 4: a few hot neurons fire on most inputs):
  f_i = min(cap, c * rank_i^-alpha), rank a seeded random permutation of
  1..ffn, with c found by bisection so that mean(f) equals the target.
* The gated projection's bias makes neuron i fire with probability f_i for
  x ~ N(0, I): its pre-activation W_i.x has std sigma_i = ||W_i||_2 (taken in
  float64 of the fp16-rounded row), so b_i = sigma_i * Phi^-1(f_i) gives
  P(W_i.x + b_i > 0) = f_i exactly.
* The predictor output bias c_p is calibrated the same way, from moments
  only: with s_k = ||W_p1_k||, h_k = ReLU(W_p1_k.x) has mean s_k/sqrt(2 pi)
  and the pairwise second moments of the degree-1 arc-cosine kernel
  (Cho & Saul 2009): E[h_k h_j] = s_k s_j (sin t + (pi - t) cos t) / (2 pi),
  cos t = <W_p1_k, W_p1_j> / (s_k s_j).  Treating W_p2_i.h as Gaussian with
  that mean mu_i and variance v_i, c_p_i = -mu_i + sqrt(v_i) Phi^-1(f_i)
  makes the predicted firing rate approximately f_i.  This is a property of
  the weights alone; no token passes through the predictor here.

Random numbers come from torch generators seeded by ``sub_seed`` so every
tensor of every layer has its own reproducible stream, on the CPU or on a GPU.
"""
from __future__ import annotations

import math
import zlib
from typing import Dict, Optional

import numpy as np
import torch

from .configs import LayerSpec


def sub_seed(base: int, layer: int, name: str) -> int:
    """Stable 63-bit seed for one tensor of one layer."""
    h = zlib.crc32(f"{base}/{layer}/{name}".encode())
    return (int(base) * 1_000_003 + int(layer) * 7919 + h) & 0x7FFF_FFFF_FFFF_FFFF


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _randn_half(shape, std, device, seed) -> torch.Tensor:
    g = _gen(device, seed)
    t = torch.randn(*shape, generator=g, device=device, dtype=torch.float32)
    t.mul_(std)
    return t.half()


def firing_rates(ffn: int, alpha: float, mean_f: float, cap: float, seed: int):
    """Per-neuron target firing rates f (float64 numpy) and the scale c."""
    g = _gen("cpu", seed)
    rank = torch.randperm(ffn, generator=g).numpy().astype(np.float64) + 1.0
    base = rank ** (-alpha)
    lo, hi = 0.0, 1.0
    while np.minimum(cap, hi * base).mean() < mean_f:
        hi *= 2.0
    for _ in range(200):
        mid = 0.5 * (lo + hi)
        if np.minimum(cap, mid * base).mean() < mean_f:
            lo = mid
        else:
            hi = mid
    c = 0.5 * (lo + hi)
    return np.minimum(cap, c * base), c


def _ndtri(p: torch.Tensor) -> torch.Tensor:
    return torch.special.ndtri(p)


def _row_norms(W: torch.Tensor, chunk: int = 4096) -> torch.Tensor:
    out = torch.empty(W.shape[0], dtype=torch.float64, device=W.device)
    for i in range(0, W.shape[0], chunk):
        out[i:i + chunk] = W[i:i + chunk].double().pow(2).sum(1).sqrt()
    return out


def predictor_logit_moments(W_p1: torch.Tensor, W_p2: torch.Tensor):
    """Mean and variance of W_p2_i . h over x ~ N(0, I), h = ReLU(W_p1 x),
    from the first- and second-order arc-cosine moments of ReLU features."""
    A = W_p1.double()
    s = A.pow(2).sum(1).sqrt()                                  # [r]
    G = A @ A.T
    cos_t = (G / torch.outer(s, s)).clamp(-1.0, 1.0)
    t = torch.arccos(cos_t)
    E_hh = torch.outer(s, s) * (torch.sin(t) + (math.pi - t) * cos_t) / (2.0 * math.pi)
    E_h = s / math.sqrt(2.0 * math.pi)
    C = E_hh - torch.outer(E_h, E_h)
    mu = torch.empty(W_p2.shape[0], dtype=torch.float64, device=W_p2.device)
    var = torch.empty_like(mu)
    for i in range(0, W_p2.shape[0], 8192):
        B = W_p2[i:i + 8192].double()
        mu[i:i + 8192] = B @ E_h
        var[i:i + 8192] = ((B @ C) * B).sum(1)
    return mu, var


def _calibrated_predictor_bias(W_p1: torch.Tensor, W_p2: torch.Tensor,
                               f: torch.Tensor) -> torch.Tensor:
    mu, var = predictor_logit_moments(W_p1, W_p2)
    return (-mu + var.clamp_min(0).sqrt() * _ndtri(f)).float()


def make_layer(spec: LayerSpec, base_seed: int, layer: int = 0,
               device="cpu") -> Dict[str, Optional[torch.Tensor]]:
    """One synthetic layer in model space (PyTorch Linear weight layouts).

    Returns W_up [ffn,d], W_gate [ffn,d] or None, b [ffn] fp32 (bias of the
    gated projection: up for ReLU, gate for ReGLU / SwiGLU), W_down [d,ffn],
    W_p1 [r,d], W_p2 [ffn,r], c_p [ffn] fp32 or None, and f [ffn] float64
    (the target firing rates, on the CPU).
    """
    d, ffn, r = spec.d, spec.ffn, spec.rank
    S = lambda name: sub_seed(base_seed, layer, name)  # noqa: E731
    W_up = _randn_half((ffn, d), spec.w_std, device, S("W_up"))
    W_gate = _randn_half((ffn, d), spec.w_std, device, S("W_gate")) if spec.act in ("reglu", "swiglu") else None
    W_down = _randn_half((d, ffn), spec.w_std, device, S("W_down"))
    W_p1 = _randn_half((r, d), spec.wp_std, device, S("W_p1"))
    W_p2 = _randn_half((ffn, r), spec.wp_std, device, S("W_p2"))
    f_np, _ = firing_rates(ffn, spec.alpha, spec.mean_f, spec.f_cap, S("rates"))
    f = torch.from_numpy(f_np).to(device)
    gated = W_gate if W_gate is not None else W_up
    b = (_row_norms(gated) * _ndtri(f)).float()
    c_p = None
    if spec.predictor_bias == "calibrated":
        c_p = _calibrated_predictor_bias(W_p1, W_p2, f)
    elif spec.predictor_bias != "none":
        raise ValueError(spec.predictor_bias)
    return dict(W_up=W_up, W_gate=W_gate, b=b, W_down=W_down, W_p1=W_p1,
                W_p2=W_p2, c_p=c_p, f=torch.from_numpy(f_np), act=spec.act)


def make_tokens(d: int, n: int, seed: int, device="cpu") -> torch.Tensor:
    """n decode-token inputs x ~ N(0, I), fp16 [n, d]."""
    return _randn_half((n, d), 1.0, device, seed)


# ---------------------------------------------------------------------------
# Exact-arithmetic mode: small-integer data scaled by powers of two, so every
# fp32 partial sum of every dot product is exact in any order (the caller
# checks the realised magnitude bound).  Weights take values {-1,0,+1}/8 with
# P(nonzero) = p_nz, tokens {-1,0,+1}, biases small integers, c_p multiples of
# 1/64 (the grid of W_p2.h), so exact ties l == 0 occur.
# ---------------------------------------------------------------------------

def _ternary(shape, p_nz, scale, seed) -> torch.Tensor:
    g = _gen("cpu", seed)
    u = torch.rand(*shape, generator=g)
    sgn = torch.randint(0, 2, shape, generator=g).float() * 2 - 1
    t = torch.where(u < p_nz, sgn, torch.zeros(()))
    return (t * scale).half()


def make_exact_layer(d: int, ffn: int, r: int, act: str = "relu", seed: int = 7,
                     p_nz: float = 0.25) -> Dict[str, Optional[torch.Tensor]]:
    S = lambda name: sub_seed(seed, 0, "exact/" + name)  # noqa: E731
    W_up = _ternary((ffn, d), p_nz, 0.125, S("W_up"))
    W_gate = _ternary((ffn, d), p_nz, 0.125, S("W_gate")) if act in ("reglu", "swiglu") else None
    W_down = _ternary((d, ffn), p_nz, 0.125, S("W_down"))
    W_p1 = _ternary((r, d), p_nz, 0.125, S("W_p1"))
    W_p2 = _ternary((ffn, r), p_nz, 0.125, S("W_p2"))
    g = _gen("cpu", S("b"))
    b = torch.randint(-3, 2, (ffn,), generator=g).float()
    c_p = (torch.randint(-8, 9, (ffn,), generator=g).float() / 64.0)
    return dict(W_up=W_up, W_gate=W_gate, b=b, W_down=W_down, W_p1=W_p1,
                W_p2=W_p2, c_p=c_p, f=None, act=act)


def make_exact_tokens(d: int, n: int, seed: int) -> torch.Tensor:
    return _ternary((n, d), 0.6, 1.0, sub_seed(seed, 0, "exact/x"))
