"""Float64 reference of the predictor-gated, neuron-aware sparse FFN.

Test infrastructure: only tests, the smoke check and the benchmark's CPU
baseline use this module.  It shares no code with the CUDA library.

Everything is computed in float64 from the fp16 / fp32 inputs exactly as
given.  Citations name the page "PowerInfer: Fast Large Language Model Serving
with a Consumer-grade GPU" (egguo-blog reading report) and its sections.
"""
from __future__ import annotations

from dataclasses import dataclass, replace
from typing import Dict, Optional

import numpy as np

_U32 = 2.0 ** -24          # unit roundoff of IEEE binary32 (round to nearest)


def _np(t):
    if t is None:
        return None
    if hasattr(t, "detach"):
        t = t.detach().cpu().numpy()
    return np.asarray(t)


def _f64(a):
    return None if a is None else np.asarray(a, dtype=np.float64)


def _gamma(n: int) -> float:
    """Higham's gamma_n = n u / (1 - n u) for binary32."""
    return n * _U32 / (1.0 - n * _U32)


@dataclass
class OracleLayer:
    """One FFN layer in the index space it is given (model space or permuted).

    act     "relu", "reglu" or "swiglu"
    W_up    fp16 [ffn, d]   up projection (PyTorch Linear(d, ffn).weight layout)
    W_gate  fp16 [ffn, d]   gate projection (ReGLU only)
    b       fp32 [ffn]      bias of the gated projection (up for ReLU, gate for ReGLU / SwiGLU)
    W_down  fp16 [d, ffn]   down projection (Linear(ffn, d).weight layout)
    W_p1    fp16 [r, d]     predictor first layer
    W_p2    fp16 [ffn, r]   predictor second layer
    c_p     fp32 [ffn]      predictor output bias (None: zero)
    """
    act: str
    W_up: np.ndarray
    W_gate: Optional[np.ndarray]
    b: np.ndarray
    W_down: np.ndarray
    W_p1: np.ndarray
    W_p2: np.ndarray
    c_p: Optional[np.ndarray]

    @classmethod
    def from_tensors(cls, t: Dict) -> "OracleLayer":
        return cls(act=t["act"], W_up=_np(t["W_up"]), W_gate=_np(t.get("W_gate")),
                   b=_np(t["b"]), W_down=_np(t["W_down"]), W_p1=_np(t["W_p1"]),
                   W_p2=_np(t["W_p2"]), c_p=_np(t.get("c_p")))

    @property
    def d(self) -> int:
        return self.W_up.shape[1]

    @property
    def ffn(self) -> int:
        return self.W_up.shape[0]

    @property
    def rank(self) -> int:
        return self.W_p1.shape[0]


# --------------------------------------------------------------------------
# Predictor (section 2.3, core module 3 "adaptive predictor": a small MLP per
# layer that predicts which neurons will fire; here one hidden ReLU layer of
# width r and no hidden bias, thresholded at sigmoid(l) > 0.5, i.e. l > 0).
# --------------------------------------------------------------------------

def predictor_hidden(L: OracleLayer, x) -> np.ndarray:
    """h = max(0, W_p1 x) for each token row of x [B, d] -> [B, r]."""
    x = _f64(x).reshape(-1, L.d)
    return np.maximum(0.0, x @ _f64(L.W_p1).T)


def predictor_logits(L: OracleLayer, h) -> np.ndarray:
    """l = W_p2 h + c_p -> [B, ffn]."""
    l = _f64(h) @ _f64(L.W_p2).T
    if L.c_p is not None:
        l = l + _f64(L.c_p)[None, :]
    return l


def predicted_mask(l) -> np.ndarray:
    """Neuron i is predicted active iff sigmoid(l_i) > 0.5, i.e. l_i > 0.

    A logit of exactly zero (either sign) counts as inactive.
    """
    return np.asarray(l) > 0.0


def active_union(mask) -> np.ndarray:
    """Ascending list of the neurons predicted active for any token of the batch.

    With a batch the operators must cover every token's active neurons, so the
    set is the union over the batch (section 4.4, limitation 3: the speed-up
    shrinks with batch size because this union grows).
    """
    m = np.asarray(mask, dtype=bool).reshape(-1, np.asarray(mask).shape[-1])
    return np.flatnonzero(m.any(axis=0)).astype(np.int64)


def logit_error_bound(L: OracleLayer, x, h=None, split: bool = False) -> np.ndarray:
    """Bound on |l_fp32 - l| for a GPU that computes h and l in binary32.

    Products of two fp16 values are exact in binary32; a dot of n terms has
    error at most gamma_n * sum|terms| in any summation order.  With
    e_k = gamma_d sum_j |W_p1_kj x_j| >= |h32_k - h_k| (ReLU is 1-Lipschitz),
    tau_i = 2 * [gamma_{r+1} (sum_k |W_p2_ik| (h_k + e_k) + |c_i|)
                 + sum_k |W_p2_ik| e_k],
    the leading 2 being slack.  Decisions with |l_i| > tau_i are forced.

    split: the form in which h enters fp16 products as a pair h32 = hi + lo + s
    (hi = fp16(h32), lo = fp16(h32 - hi)), as on tensor cores.  Then
    |s_k| <= 2^-22 |h32_k| + 2^-25 (two fp16 roundings; the 2^-25 covers lo in
    fp16's subnormal range), the sum runs over 2r products plus c, and
    |hi| + |lo| <= |h32| (1 + 2^-10), so
    tau_i = 2 * [gamma_{2r+1} (sum_k |W_p2_ik| m_k + |c_i|) + sum_k |W_p2_ik| (e_k + s_k)]
    with m_k = (h_k + e_k)(1 + 2^-10) and s_k = 2^-22 (h_k + e_k) + 2^-25.
    """
    x = _f64(x).reshape(-1, L.d)
    if h is None:
        h = predictor_hidden(L, x)
    A1 = np.abs(_f64(L.W_p1))
    A2 = np.abs(_f64(L.W_p2))
    e = _gamma(L.d) * (np.abs(x) @ A1.T)                 # [B, r]
    cabs = 0.0 if L.c_p is None else np.abs(_f64(L.c_p))[None, :]
    if not split:
        tau = _gamma(L.rank + 1) * ((h + e) @ A2.T + cabs) + e @ A2.T
    else:
        s = fp16_pair_error_bound(h + e)
        m = (h + e) * (1.0 + 2.0 ** -10)
        tau = _gamma(2 * L.rank + 1) * (m @ A2.T + cabs) + (e + s) @ A2.T
    return 2.0 * tau


def fp16_pair_error_bound(v) -> np.ndarray:
    """Bound on |v - hi - lo| for the fp16 pair of binary32 values of magnitude
    at most |v|: the two fp16 roundings leave at most 2^-22 |v| relative, and
    at most 2^-25 absolute once lo falls in fp16's subnormal range (spacing
    2^-24)."""
    return 2.0 ** -22 * np.abs(_f64(v)) + 2.0 ** -25


def fp16_pair(v) -> tuple:
    """The fp16 pair (hi, lo) of binary32 values v: hi = fp16(v), lo = fp16(v - hi),
    v - hi formed in binary32 (exact: hi is v rounded to a coarser grid)."""
    v32 = np.asarray(v, dtype=np.float32)
    hi = v32.astype(np.float16)
    lo = (v32 - hi.astype(np.float32)).astype(np.float16)
    return hi, lo


# --------------------------------------------------------------------------
# Neuron-aware sparse FFN (section 2.3, core module 4: a sparse matrix-vector
# product that works directly on individual neurons).  For each neuron i of
# the set S: ReLU   a_i = max(0, W_up_i . x + b_i)
#            ReGLU  a_i = max(0, W_gate_i . x + b_i) * (W_up_i . x)
#            SwiGLU a_i = SiLU(W_gate_i . x + b_i) * (W_up_i . x)
# and y = sum over i in S (ascending) of a_i * W_down[:, i].  For SwiGLU the
# set is a pruning choice (section 2.3, variable table: neurons that can be
# skipped with a small effect on the output), so the sum over S differs from
# the dense FFN by the skipped neurons' terms.
# --------------------------------------------------------------------------

def silu(z) -> np.ndarray:
    """SiLU(z) = z * sigmoid(z) = z / (1 + e^-z), written per sign so that no
    exponential overflows: z / (1 + e^-z) for z >= 0, z e^z / (1 + e^z) below."""
    z = _f64(z)
    e = np.exp(-np.abs(z))                       # in (0, 1]
    return np.where(z >= 0, z / (1.0 + e), z * e / (1.0 + e))

def _rowdots(W16: np.ndarray, rows: np.ndarray, xb: np.ndarray, chunk: int = 512) -> np.ndarray:
    """W[rows] . xb in float64, each row summed on its own (chunking over rows
    changes no arithmetic)."""
    out = np.empty(rows.shape[0], dtype=np.float64)
    for s in range(0, rows.shape[0], chunk):
        blk = _f64(W16[rows[s:s + chunk]])
        out[s:s + chunk] = (blk * xb[None, :]).sum(axis=1)
    return out


def ffn_activations(L: OracleLayer, x, S) -> np.ndarray:
    """a [B, |S|] for the neurons of S, in the order S lists them."""
    x = _f64(x).reshape(-1, L.d)
    S = np.asarray(S, dtype=np.int64)
    b = _f64(L.b)[S]
    a = np.empty((x.shape[0], S.shape[0]), dtype=np.float64)
    for t in range(x.shape[0]):
        if L.act == "relu":
            a[t] = np.maximum(0.0, _rowdots(L.W_up, S, x[t]) + b)
        elif L.act == "reglu":
            g = np.maximum(0.0, _rowdots(L.W_gate, S, x[t]) + b)
            a[t] = g * _rowdots(L.W_up, S, x[t])
        elif L.act == "swiglu":
            g = silu(_rowdots(L.W_gate, S, x[t]) + b)
            a[t] = g * _rowdots(L.W_up, S, x[t])
        else:
            raise ValueError(L.act)
    return a


def ffn_output(L: OracleLayer, S, a) -> np.ndarray:
    """y [B, d] = sum over k (in the order of S) of a[:, k] * W_down[:, S[k]]."""
    S = np.asarray(S, dtype=np.int64)
    a = _f64(a)
    if a.ndim == 1:
        a = a[None, :]
    y = np.zeros((a.shape[0], L.d), dtype=np.float64)
    for s in range(0, S.shape[0], 1024):
        cols = _f64(L.W_down[:, S[s:s + 1024]]).T          # [chunk, d] rows of W_down^T
        for k in range(cols.shape[0]):
            y += a[:, s + k:s + k + 1] * cols[k][None, :]
    return y


def sparse_ffn(L: OracleLayer, x, S) -> np.ndarray:
    """The FFN restricted to the neurons in S (ascending), float64."""
    S = np.asarray(S, dtype=np.int64)
    return ffn_output(L, S, ffn_activations(L, x, S))


def dense_ffn(L: OracleLayer, x) -> np.ndarray:
    """The ordinary dense FFN: the same sum over every neuron."""
    return sparse_ffn(L, x, np.arange(L.ffn))


def exact_mask(L: OracleLayer, x):
    """True activation pattern: (mask [B, ffn], z [B, ffn]).

    ReLU sparsity is the share of neurons whose activation is exactly zero
    (section 2.3, variable table, "sparsity"); a neuron is active iff the
    pre-activation of its gated projection is > 0 (up for ReLU, gate for
    ReGLU).  For SwiGLU, whose activation is never exactly zero, the same
    rule (the gate on SiLU's positive branch) serves the profile that orders
    neurons hot-first.
    """
    x = _f64(x).reshape(-1, L.d)
    Wg = L.W_gate if L.act in ("reglu", "swiglu") else L.W_up
    z = x @ _f64(Wg).T + _f64(L.b)[None, :]
    return z > 0.0, z


def preact_error_bound(L: OracleLayer, x) -> np.ndarray:
    """Bound on |z_fp32 - z| for the gated pre-activation computed in binary32."""
    x = _f64(x).reshape(-1, L.d)
    Wg = L.W_gate if L.act in ("reglu", "swiglu") else L.W_up
    s = np.abs(x) @ np.abs(_f64(Wg)).T + np.abs(_f64(L.b))[None, :]
    return 2.0 * _gamma(L.d + 1) * s


def predicted_forward(L: OracleLayer, x) -> Dict[str, np.ndarray]:
    """The whole path for one batch: predictor, union set, sparse FFN.
    tau is the band of the bound's fp16-pair form (split=True), which also
    covers the plain binary32 form: a GPU may compute the logits either way."""
    x = _f64(x).reshape(-1, L.d)
    h = predictor_hidden(L, x)
    l = predictor_logits(L, h)
    mask = predicted_mask(l)
    S = active_union(mask)
    y = sparse_ffn(L, x, S)
    return dict(h=h, l=l, mask=mask, S=S, y=y, tau=logit_error_bound(L, x, h, split=True))


# --------------------------------------------------------------------------
# Offline profile and hot-first order (section 2.3, core module 1 "LLM
# profiler": per-neuron activation counts over a corpus; variable table:
# neuron impact v_i = f_i, the activation frequency; hot neurons are the few
# that carry 80% of activations).
# --------------------------------------------------------------------------

def profile_counts(L: OracleLayer, X, chunk: int = 256):
    """Per-neuron count of tokens on which the neuron fires, plus the count of
    (token, neuron) pairs whose decision lies inside the binary32 band."""
    X = _f64(X).reshape(-1, L.d)
    counts = np.zeros(L.ffn, dtype=np.int64)
    band = np.zeros(L.ffn, dtype=np.int64)
    for s in range(0, X.shape[0], chunk):
        xb = X[s:s + chunk]
        m, z = exact_mask(L, xb)
        tau = preact_error_bound(L, xb)
        counts += m.sum(axis=0)
        band += (np.abs(z) <= tau).sum(axis=0)
    return counts, band


def hot_first_order(counts) -> np.ndarray:
    """perm with perm[k] = the neuron placed at position k: counts descending,
    ties by ascending neuron index."""
    c = np.asarray(counts, dtype=np.int64)
    return np.argsort(-c, kind="stable").astype(np.int64)


def permute_layer(L: OracleLayer, perm) -> OracleLayer:
    """The same layer with neuron k of the result = neuron perm[k] of L."""
    p = np.asarray(perm, dtype=np.int64)
    return replace(
        L,
        W_up=L.W_up[p],
        W_gate=None if L.W_gate is None else L.W_gate[p],
        b=L.b[p],
        W_down=L.W_down[:, p],
        W_p2=L.W_p2[p],
        c_p=None if L.c_p is None else L.c_p[p],
    )
