"""SwiGLU layers (a_i = SiLU(gate) * up over the predicted set) on the GPU
against the float64 oracle: the decode step at 1-2 tokens, the tensor-core
path, the standalone operators, FP8 rows and the activation profile."""
import numpy as np
import pytest
import torch

from oracle import ffn as O
from oracle import quant as Q
from tests.gpu_helpers import check_union_set, check_y, oracle_y_for_valid_set, stored_oracle, to_dev
from workload import LayerSpec, make_layer, make_tokens

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pi():
    import __graft_entry__
    __graft_entry__.build()
    import activation_sparse_rank_gb300 as pi
    return pi


def _check_forward(layer, L, x, B):
    y, idx, count = layer.forward(x.cuda())
    torch.cuda.synchronize()
    S = idx[: int(count.item())].cpu().numpy().astype(np.int64)
    r = O.predicted_forward(L, x)
    band = check_union_set(S, r["l"], r["tau"])
    check_y(y.cpu().numpy(), oracle_y_for_valid_set(L, x, S))
    return S, band


@pytest.mark.parametrize("d,ffn,r", [(1024, 4096, 64), (2048, 3000, 40), (8192, 2000, 128)])
@pytest.mark.parametrize("B", [1, 2, 3, 8, 32])
def test_forward(pi, d, ffn, r, B):
    t = make_layer(LayerSpec(d=d, ffn=ffn, rank=r, act="swiglu", mean_f=0.5), 51, 0)
    layer = pi.Layer.from_dict(to_dev(t))
    assert layer.act == "swiglu"
    L = stored_oracle(layer, t)
    for rep in range(2):
        _check_forward(layer, L, make_tokens(d, B, seed=60 + rep), B)
    assert layer.device_status() == 0


@pytest.mark.parametrize("B", [1, 2, 5])
def test_standalone_operators_and_generic_batch_path(pi, B):
    # d = 1032 is not a multiple of 64: batches of 3+ take the generic kernels
    d, ffn, r = 1032, 1500, 32
    t = make_layer(LayerSpec(d=d, ffn=ffn, rank=r, act="swiglu", mean_f=0.5), 52, 0)
    layer = pi.Layer.from_dict(to_dev(t))
    L = stored_oracle(layer, t)
    x = make_tokens(d, B, seed=7)
    S = np.flatnonzero(np.random.default_rng(3).random(ffn) < 0.4).astype(np.int32)
    y = layer.sparse_ffn(x.cuda(), torch.from_numpy(S).cuda(),
                         torch.tensor([S.size], dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    check_y(y.cpu().numpy(), O.sparse_ffn(L, x, S.astype(np.int64)))
    yd = layer.dense_ref(x.cuda())
    torch.cuda.synchronize()
    check_y(yd.cpu().numpy(), O.dense_ffn(L, x))
    _check_forward(layer, L, x, B)


def test_fp8_rows(pi):
    d, ffn, r = 2048, 6000, 64
    t = make_layer(LayerSpec(d=d, ffn=ffn, rank=r, act="swiglu", mean_f=0.5), 53, 0)
    layer = pi.Layer.from_dict(to_dev(t), rows="fp8")
    L8 = Q.fp8_layer(stored_oracle(layer, t))
    for B in (1, 2):
        _check_forward(layer, L8, make_tokens(d, B, seed=70 + B), B)


def test_profile_counts_use_the_gate(pi):
    d, ffn, r = 512, 768, 16
    t = make_layer(LayerSpec(d=d, ffn=ffn, rank=r, act="swiglu", mean_f=0.5), 54, 0)
    X = make_tokens(d, 300, seed=9)
    counts = pi.profile_activations(to_dev(t), X.cuda()).cpu().numpy()
    ref, band = O.profile_counts(O.OracleLayer.from_tensors(t), X)
    assert np.all(np.abs(counts - ref) <= band)
