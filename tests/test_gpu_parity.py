"""Parity of the CUDA library (through the C ABI) with the float64 CPU oracle.

Sizes span several CTA chunks and ragged tails; all inputs are seeded.
"""
import numpy as np
import pytest
import torch

from oracle import ffn as O
from tests.gpu_helpers import (check_union_set, check_y, dealt_order, oracle_y_for_valid_set,
                               sm_count, stored_oracle, to_dev)
from workload import LayerSpec, make_layer, make_tokens
from workload.gen import make_exact_layer, make_exact_tokens

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pi():
    import __graft_entry__
    __graft_entry__.build()
    import activation_sparse_rank_gb300 as pi
    return pi


def _layer(spec, seed):
    t = make_layer(spec, seed)
    return t, O.OracleLayer.from_tensors(t)


SHAPES = [
    # d, ffn, rank, act
    (1024, 4096, 64, "relu"),      # single OPT-style layer
    (520, 1000, 24, "relu"),       # ragged everywhere
    (4096, 2048, 256, "relu"),
    (8192, 1024, 512, "reglu"),
    (12288, 768, 1024, "relu"),
    (16384, 512, 64, "reglu"),
]


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("B", [1, 3, 9])
def test_predict(pi, shape, B):
    d, ffn, r, act = shape
    t, _ = _layer(LayerSpec(d=d, ffn=ffn, rank=r, act=act, mean_f=0.1), seed=d + B)
    x = make_tokens(d, B, seed=5 + B)
    layer = pi.Layer.from_dict(to_dev(t))
    L = stored_oracle(layer, t)
    mask, logits = layer.predict(x.cuda(), want_logits=True)
    torch.cuda.synchronize()
    l_gpu = logits.cpu().numpy().astype(np.float64)
    m_gpu = mask.cpu().numpy().astype(bool)
    h = O.predictor_hidden(L, x)
    l = O.predictor_logits(L, h)
    tau = O.logit_error_bound(L, x, h, split=B > 2)   # B > 2: tensor-core form
    assert (np.abs(l_gpu - l) <= tau).all()
    np.testing.assert_array_equal(m_gpu, l_gpu > 0)
    forced = np.abs(l) > tau
    np.testing.assert_array_equal(m_gpu[forced], (l > 0)[forced])
    assert layer.device_status() == 0


@pytest.mark.parametrize("ffn", [1, 15, 16, 1000, 16391, 49152])
@pytest.mark.parametrize("B", [1, 4])
def test_compact(pi, ffn, B):
    rng = np.random.default_rng(ffn + B)
    d, r = 64, 8
    t, _ = _layer(LayerSpec(d=d, ffn=ffn, rank=r), seed=3)
    layer = pi.Layer.from_dict(to_dev(t))
    for density in (0.0, 0.02, 0.5, 1.0):
        m = (rng.random((B, ffn)) < density).astype(np.uint8)
        idx = torch.full((ffn + 3,), -7, dtype=torch.int32, device="cuda")
        idx, count = layer.compact(torch.from_numpy(m).cuda(), idx=idx)
        torch.cuda.synchronize()
        n = int(count.item())
        S = O.active_union(m)
        assert n == S.size
        got = idx.cpu().numpy()
        np.testing.assert_array_equal(got[:n], S)
        assert (got[n:] == -7).all()          # entries past count untouched


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("B", [1, 2, 3, 5])
def test_sparse_ffn(pi, shape, B):
    d, ffn, r, act = shape
    t, _ = _layer(LayerSpec(d=d, ffn=ffn, rank=r, act=act, mean_f=0.12), seed=7 * d + B)
    x = make_tokens(d, B, seed=11 + B)
    layer = pi.Layer.from_dict(to_dev(t))
    L = stored_oracle(layer, t)
    S = O.predicted_forward(L, x)["S"]             # the oracle's own set as input
    idx = torch.from_numpy(S.astype(np.int32)).cuda()
    count = torch.tensor([S.size], dtype=torch.int32, device="cuda")
    y = layer.sparse_ffn(x.cuda(), idx, count)
    y2 = layer.sparse_ffn(x.cuda(), idx, count)
    torch.cuda.synchronize()
    check_y(y.cpu().numpy(), O.sparse_ffn(L, x, S))
    assert torch.equal(y, y2), "two runs must be bitwise identical"
    assert layer.device_status() == 0


@pytest.mark.parametrize("shape", SHAPES[:4])
@pytest.mark.parametrize("B", [1, 4])
def test_dense_ref_and_exact_mask(pi, shape, B):
    d, ffn, r, act = shape
    t, _ = _layer(LayerSpec(d=d, ffn=ffn, rank=r, act=act, mean_f=0.1), seed=13 * d + B)
    x = make_tokens(d, B, seed=17 + B)
    layer = pi.Layer.from_dict(to_dev(t))
    L = stored_oracle(layer, t)
    yd = layer.dense_ref(x.cuda())
    m, _ = O.exact_mask(L, x)
    S = O.active_union(m)
    ys = layer.sparse_ffn(x.cuda(), torch.from_numpy(S.astype(np.int32)).cuda(),
                          torch.tensor([S.size], dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    y_dense = O.dense_ffn(L, x)
    check_y(yd.cpu().numpy(), y_dense)
    check_y(ys.cpu().numpy(), y_dense)      # sparse over the exact mask == dense


@pytest.mark.parametrize("act", ["relu", "reglu"])
def test_rows_outside_set_are_never_read(pi, act):
    d, ffn, r = 2048, 4096, 64
    t, L = _layer(LayerSpec(d=d, ffn=ffn, rank=r, act=act, mean_f=0.1), seed=19)
    x = make_tokens(d, 1, seed=23).cuda()
    clean = pi.Layer.from_dict(to_dev(t))
    _, idx, count = clean.forward(x)
    torch.cuda.synchronize()
    S = idx[:int(count.item())].cpu().numpy()
    y0 = clean.sparse_ffn(x, torch.from_numpy(S.astype(np.int32)).cuda(), count)
    out = torch.from_numpy(clean.perm()[np.setdiff1d(np.arange(ffn), S)].astype(np.int64))
    p = dict(t)
    p["W_up"] = t["W_up"].clone(); p["W_up"][out] = float("nan")
    p["W_down"] = t["W_down"].clone(); p["W_down"][:, out] = float("inf")
    if act == "reglu":
        p["W_gate"] = t["W_gate"].clone(); p["W_gate"][out] = float("nan")
    poisoned = pi.Layer.from_dict(to_dev(p))
    idx_t = torch.from_numpy(S.astype(np.int32)).cuda()
    y1 = poisoned.sparse_ffn(x, idx_t, count)
    torch.cuda.synchronize()
    assert torch.isfinite(y1).all()
    assert torch.equal(y0, y1)


@pytest.mark.parametrize("act", ["relu", "reglu"])
@pytest.mark.parametrize("B", [1, 2, 3])
def test_exact_arithmetic_bitwise(pi, act, B):
    """Integer-grid data: every binary32 sum is exact, so the GPU must match the
    oracle bit for bit (set and output) whatever its summation order."""
    t = make_exact_layer(1024, 2048, 64, act=act, seed=5)
    X = make_exact_tokens(1024, B, seed=6)
    layer = pi.Layer.from_dict(to_dev(t))
    L = stored_oracle(layer, t)
    y, idx, count = layer.forward(X.cuda())
    torch.cuda.synchronize()
    r = O.predicted_forward(L, X)
    n = int(count.item())
    np.testing.assert_array_equal(idx[:n].cpu().numpy(), r["S"])
    a = O.ffn_activations(L, X, r["S"])
    assert ((np.abs(a) @ np.abs(L.W_down[:, r["S"]].astype(np.float64)).T).max() * 512) < 2 ** 24
    np.testing.assert_array_equal(y.cpu().numpy().astype(np.float64), r["y"])


def test_empty_set_and_bad_inputs(pi):
    d, ffn, r = 1024, 4096, 64
    t, _ = _layer(LayerSpec(d=d, ffn=ffn, rank=r), seed=29)
    layer = pi.Layer.from_dict(to_dev(t))
    L = stored_oracle(layer, t)
    x = make_tokens(d, 1, seed=31)
    xc = x.cuda()
    idx = torch.arange(ffn, dtype=torch.int32, device="cuda")
    y = layer.sparse_ffn(xc, idx, torch.tensor([0], dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    assert (y == 0).all() and layer.device_status() == 0
    # count beyond ffn is clamped and flagged
    y = layer.sparse_ffn(xc, idx, torch.tensor([ffn + 10], dtype=torch.int32, device="cuda"))
    assert layer.device_status() == 5
    check_y(y.cpu().numpy(), O.dense_ffn(L, x))
    # out-of-range entries are skipped and flagged
    S = np.array([3, 17, ffn + 5, 99, -2, 4000], dtype=np.int32)
    y = layer.sparse_ffn(xc, torch.from_numpy(S).cuda(), torch.tensor([6], dtype=torch.int32, device="cuda"))
    assert layer.device_status() == 5
    check_y(y.cpu().numpy(), O.sparse_ffn(L, x, np.array([3, 17, 99, 4000])))
    assert layer.device_status() == 0


def test_host_side_rejections_leave_the_gpu_untouched(pi):
    """A bad permutation, a workspace that is too small and a batch beyond the
    limit are refused on the host with an error code; the layer and the device
    stay usable."""
    d, ffn, r = 256, 512, 16
    t, _ = _layer(LayerSpec(d=d, ffn=ffn, rank=r, mean_f=0.2), seed=41)
    td = to_dev(t)
    for bad in (np.r_[np.arange(ffn - 1), 0],          # a duplicate
                np.r_[np.arange(ffn - 1), ffn],        # out of range
                np.arange(ffn - 1)):                   # too short is read as ffn entries: pad with -1
        perm = bad if bad.size == ffn else np.r_[bad, -1]
        with pytest.raises(pi.PiError) as e:
            pi.Layer.from_dict(td, perm=perm)
        assert e.value.status == 1                     # PI_ERR_INVALID_ARG
    layer = pi.Layer.from_dict(td)
    x = make_tokens(d, 1, seed=1).cuda()
    small = torch.empty(64, dtype=torch.uint8, device="cuda")
    with pytest.raises(pi.PiError) as e:
        layer.forward(x, ws=small)
    assert e.value.status == 1
    with pytest.raises(pi.PiError) as e:
        layer.forward(make_tokens(d, 129, seed=2).cuda())   # B > PI_MAX_BATCH
    assert e.value.status == 1
    y, idx, count = layer.forward(x)                   # still works
    torch.cuda.synchronize()
    assert torch.isfinite(y).all() and layer.device_status() == 0


def test_permuted_layer(pi):
    d, ffn, r = 2048, 8192, 128
    t, L = _layer(LayerSpec(d=d, ffn=ffn, rank=r, mean_f=0.1), seed=37)
    perm = np.random.default_rng(4).permutation(ffn).astype(np.int32)
    layer = pi.Layer.from_dict(to_dev(t), perm=perm)
    stored = layer.perm()
    np.testing.assert_array_equal(stored, dealt_order(perm, sm_count()))
    identity = pi.Layer.from_dict(to_dev(t)).perm()
    np.testing.assert_array_equal(identity, dealt_order(np.arange(ffn), sm_count()))
    perm = stored
    P = O.permute_layer(L, perm)
    X = make_tokens(d, 4, seed=41)
    for b in range(4):
        x = X[b:b + 1]
        y, idx, count = layer.forward(x.cuda())
        torch.cuda.synchronize()
        S = idx[:int(count.item())].cpu().numpy().astype(np.int64)
        rP = O.predicted_forward(P, x)
        check_union_set(S, rP["l"], rP["tau"])
        y_ref = oracle_y_for_valid_set(P, x, S)
        check_y(y.cpu().numpy(), y_ref)
        # and the same y as the unpermuted model, within rounding
        check_y(y.cpu().numpy(), O.sparse_ffn(L, x, np.sort(perm[S])))


@pytest.mark.parametrize("B", [1, 2, 4])
def test_layer_forward_single_opt_layer(pi, B):
    """The single OPT-style layer workload: d=1024, ffn=4096, r=64, 64 tokens."""
    t, _ = _layer(LayerSpec(d=1024, ffn=4096, rank=64, mean_f=0.10), seed=1001)
    layer = pi.Layer.from_dict(to_dev(t))
    L = stored_oracle(layer, t)
    X = make_tokens(1024, 64, seed=1001)
    band = 0
    for s in range(0, 64, B):
        x = X[s:s + B]
        y, idx, count = layer.forward(x.cuda())
        torch.cuda.synchronize()
        S = idx[:int(count.item())].cpu().numpy().astype(np.int64)
        r = O.predicted_forward(L, x)
        band += check_union_set(S, r["l"], r["tau"])
        check_y(y.cpu().numpy(), oracle_y_for_valid_set(L, x, S))
    assert layer.device_status() == 0


def test_profile_counts(pi):
    d, ffn, r = 1024, 4096, 64
    t, L = _layer(LayerSpec(d=d, ffn=ffn, rank=r, mean_f=0.1), seed=43)
    X = make_tokens(d, 700, seed=47)
    counts = pi.profile_activations(to_dev(t), X.cuda())
    torch.cuda.synchronize()
    c_ref, band = O.profile_counts(L, X)
    assert (np.abs(counts.cpu().numpy() - c_ref) <= band).all()
    # exact-grid layer: no band, counts and hot-first order must match exactly
    te = make_exact_layer(512, 1000, 16, seed=9)
    Le = O.OracleLayer.from_tensors(te)
    Xe = make_exact_tokens(512, 333, seed=10)
    ce = pi.profile_activations(to_dev(te), Xe.cuda()).cpu().numpy()
    ce_ref, _ = O.profile_counts(Le, Xe)
    np.testing.assert_array_equal(ce, ce_ref)
    np.testing.assert_array_equal(pi.hot_first_perm(ce), O.hot_first_order(ce_ref))


@pytest.mark.parametrize("act,d,ffn,r", [("relu", 4096, 6000, 256), ("reglu", 2048, 3000, 64),
                                         ("relu", 12288, 1100, 128)])
@pytest.mark.parametrize("B", [3, 8, 16, 32, 64, 128])
def test_batched_tensor_core_path(pi, act, d, ffn, r, B):
    """Batches of 3+ run the tcgen05 gathered-tile kernels: union set of the
    batch, activations split into an fp16 pair; checked on every token."""
    t, _ = _layer(LayerSpec(d=d, ffn=ffn, rank=r, act=act, mean_f=0.1), seed=d + 7 * B)
    layer = pi.Layer.from_dict(to_dev(t))
    L = stored_oracle(layer, t)
    x = make_tokens(d, B, seed=B)
    h = O.predictor_hidden(L, x)
    S = O.active_union(O.predicted_mask(O.predictor_logits(L, h)))
    idx = torch.from_numpy(S.astype(np.int32)).cuda()
    count = torch.tensor([S.size], dtype=torch.int32, device="cuda")
    y = layer.sparse_ffn(x.cuda(), idx, count)
    y2 = layer.sparse_ffn(x.cuda(), idx, count)
    torch.cuda.synchronize()
    rows = list(range(B)) if B <= 16 else [0, 1, B // 2, B - 1]
    check_y(y.cpu().numpy()[rows], O.sparse_ffn(L, x[rows], S))
    assert torch.equal(y, y2)
    assert layer.device_status() == 0
    if B in (8, 128) and act == "relu":
        yd = layer.dense_ref(x.cuda())
        torch.cuda.synchronize()
        check_y(yd.cpu().numpy()[rows], O.dense_ffn(L, x[rows]))
