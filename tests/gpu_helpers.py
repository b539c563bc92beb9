"""Shared checks for the GPU parity tests (CUDA path vs the CPU oracle)."""
import numpy as np
import torch

from oracle import ffn as O

ABS_TOL = 2e-3      # max abs error bound on y (fp16 weights, fp32 accumulation)
REL_L2_TOL = 1e-3   # relative L2 error bound on y


def stored_oracle(layer, t: dict) -> O.OracleLayer:
    """The oracle for a GPU layer as it is stored: model-space weights put in
    the layer's storage order (pi_layer_perm), so positions line up."""
    return O.permute_layer(O.OracleLayer.from_tensors(t), layer.perm())


def to_dev(t: dict, dev="cuda"):
    return {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in t.items()}


def check_union_set(S_gpu: np.ndarray, l: np.ndarray, tau: np.ndarray) -> int:
    """S_gpu must contain every neuron some token forces active (l > tau) and
    none that every token forces inactive (l < -tau).  Returns the number of
    neurons left open by the rounding band (either decision accepted)."""
    l = np.atleast_2d(l)
    tau = np.atleast_2d(tau)
    ffn = l.shape[1]
    assert np.all(np.diff(S_gpu) > 0), "active list must be strictly ascending"
    assert S_gpu.size == 0 or (S_gpu[0] >= 0 and S_gpu[-1] < ffn)
    gpu = np.zeros(ffn, bool)
    gpu[S_gpu] = True
    forced_on = (l > tau).any(axis=0)
    forced_off = (l < -tau).all(axis=0)
    bad_on = np.flatnonzero(forced_on & ~gpu)
    bad_off = np.flatnonzero(forced_off & gpu)
    assert bad_on.size == 0, f"forced-active neurons missing: {bad_on[:10]}"
    assert bad_off.size == 0, f"forced-inactive neurons present: {bad_off[:10]}"
    return int((~forced_on & ~forced_off).sum())


def check_y(y_gpu, y_ref, abs_tol=ABS_TOL, rel_tol=REL_L2_TOL):
    y = np.asarray(y_gpu, dtype=np.float64)
    r = np.asarray(y_ref, dtype=np.float64)
    assert y.shape == r.shape
    assert np.isfinite(y).all()
    err = np.abs(y - r)
    rel = np.linalg.norm(y - r) / max(np.linalg.norm(r), 1e-30)
    assert err.max() <= abs_tol, f"max abs err {err.max():.3e} > {abs_tol}"
    assert rel <= rel_tol, f"rel-L2 err {rel:.3e} > {rel_tol}"
    return float(err.max()), float(rel)


def oracle_y_for_valid_set(L: O.OracleLayer, x, S_gpu):
    """The FFN output the method defines for the GPU's active list.  Call only
    after check_union_set has accepted that list: the list then differs from
    the oracle's own set at most on neurons inside the rounding band, where
    either decision is a correct result."""
    return O.sparse_ffn(L, x, np.asarray(S_gpu, dtype=np.int64))


def dealt_order(order, G: int) -> np.ndarray:
    """The layout a layer stores for a caller's neuron order: the k-th neuron
    of `order` goes to SM slice k % G at place k // G (slices of near-equal
    size, laid out one after another)."""
    order = np.asarray(order)
    ffn = order.shape[0]
    q, rr = divmod(ffn, G)
    out = np.empty_like(order)
    for k in range(ffn):
        c, j = k % G, k // G
        out[c * q + min(c, rr) + j] = order[k]
    return out


def sm_count() -> int:
    return torch.cuda.get_device_properties(0).multi_processor_count
