"""FP8 (E4M3) row layers on the GPU against the float64 oracle: the stored
codes and scales byte for byte, and every entry point that reads the rows
(the decode step of pi_layer_forward / pi_stack_forward at 1 and 2 tokens,
pi_sparse_ffn, pi_ffn_dense_ref, batches of 3 or more tokens) against the
FFN of the dequantised rows."""
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


SHAPES = [("relu", 1024, 4096, 64), ("reglu", 2048, 3000, 40), ("relu", 4096, 16384, 256),
          ("relu", 12288, 2000, 128)]


@pytest.mark.parametrize("act,d,ffn,r", SHAPES)
def test_stored_codes_and_scales_are_the_oracles(pi, act, d, ffn, r):
    spec = LayerSpec(d=d, ffn=ffn, rank=r, act=act, mean_f=0.1)
    t = make_layer(spec, 21, 0)
    layer = pi.Layer.from_dict(to_dev(t), rows="fp8")
    ref = Q.fp8_rows(stored_oracle(layer, t))
    mats = [("up", 0), ("down", 2)] + ([("gate", 1)] if act == "reglu" else [])
    for name, m in mats:
        codes, scales = layer.rows_fp8(m)
        torch.cuda.synchronize()
        rc, rs = ref[name]
        assert np.array_equal(scales.cpu().numpy(), rs), name
        got = codes.cpu().numpy()
        bad = np.argwhere(got != rc)
        assert bad.size == 0, f"{name}: {bad.shape[0]} codes differ, first {bad[:5]}"


@pytest.mark.parametrize("act,d,ffn,r", SHAPES)
@pytest.mark.parametrize("B", [1, 2])
def test_forward_matches_dequantised_oracle(pi, act, d, ffn, r, B):
    spec = LayerSpec(d=d, ffn=ffn, rank=r, act=act, mean_f=0.1)
    t = make_layer(spec, 22, 0)
    layer = pi.Layer.from_dict(to_dev(t), rows="fp8")
    L8 = Q.fp8_layer(stored_oracle(layer, t))
    for rep in range(2):
        x = make_tokens(d, B, seed=30 + rep)
        y = torch.empty(B, d, dtype=torch.float32, device="cuda")
        idx = torch.empty(ffn, dtype=torch.int32, device="cuda")
        count = torch.empty(1, dtype=torch.int32, device="cuda")
        layer.forward(x.cuda(), idx=idx, count=count, y=y)
        torch.cuda.synchronize()
        S = idx[: int(count.item())].cpu().numpy().astype(np.int64)
        r_ = O.predicted_forward(L8, x)            # predictor is fp16: same sets as the fp16 layer
        check_union_set(S, r_["l"], r_["tau"])
        check_y(y.cpu().numpy(), oracle_y_for_valid_set(L8, x, S))
    assert layer.device_status() == 0


def test_stack_of_fp8_layers(pi):
    n, d, ffn, r = 5, 1024, 4096, 64
    spec = LayerSpec(d=d, ffn=ffn, rank=r, mean_f=0.1)
    ts = [make_layer(spec, 23, l) for l in range(n)]
    layers = [pi.Layer.from_dict(to_dev(t), rows="fp8") for t in ts]
    x = make_tokens(d, n, seed=8).view(n, 1, d)
    y = torch.empty(n, 1, d, dtype=torch.float32, device="cuda")
    idx = torch.empty((n, ffn), dtype=torch.int32, device="cuda")
    count = torch.empty(n, dtype=torch.int32, device="cuda")
    pi.stack_forward(layers, x.cuda(), y, idx=idx, count=count)
    y2 = torch.empty_like(y)
    pi.stack_forward(layers, x.cuda(), y2, idx=idx, count=count)
    torch.cuda.synchronize()
    assert torch.equal(y, y2)                       # deterministic
    for l in range(n):
        L8 = Q.fp8_layer(stored_oracle(layers[l], ts[l]))
        S = idx[l, : int(count[l].item())].cpu().numpy().astype(np.int64)
        r_ = O.predicted_forward(L8, x[l])
        check_union_set(S, r_["l"], r_["tau"])
        check_y(y[l].cpu().numpy(), oracle_y_for_valid_set(L8, x[l], S))


@pytest.mark.parametrize("act,d,ffn,r", SHAPES)
@pytest.mark.parametrize("B", [1, 2, 3, 8, 32, 128])
def test_sparse_and_dense_operators_on_fp8_rows(pi, act, d, ffn, r, B):
    """pi_sparse_ffn over a given set and pi_ffn_dense_ref over every neuron
    read the E4M3 codes (1-2 tokens: generic CUDA-core kernels; 3 or more:
    the tensor-core kernels, which convert the codes to fp16 in shared
    memory) and match the FFN of the dequantised rows; two runs agree
    bitwise."""
    spec = LayerSpec(d=d, ffn=ffn, rank=r, act=act, mean_f=0.1)
    t = make_layer(spec, 25, 0)
    layer = pi.Layer.from_dict(to_dev(t), rows="fp8")
    L8 = Q.fp8_layer(stored_oracle(layer, t))
    x = make_tokens(d, B, seed=40 + B)
    S = np.sort(np.random.default_rng(B).choice(ffn, size=ffn // 7, replace=False)).astype(np.int64)
    idx = torch.from_numpy(S.astype(np.int32)).cuda()
    count = torch.tensor([S.size], dtype=torch.int32, device="cuda")
    y = layer.sparse_ffn(x.cuda(), idx, count)
    y2 = layer.sparse_ffn(x.cuda(), idx, count)
    yd = layer.dense_ref(x.cuda())
    torch.cuda.synchronize()
    assert torch.equal(y, y2)
    rows = list(range(B)) if B <= 3 else [0, B - 1]
    check_y(y.cpu().numpy()[rows], O.sparse_ffn(L8, x[rows], S))
    check_y(yd.cpu().numpy()[rows], O.dense_ffn(L8, x[rows]))
    assert layer.device_status() == 0


@pytest.mark.parametrize("act,d,ffn,r", [("reglu", 2048, 3000, 128), ("relu", 4096, 20000, 256),
                                         ("swiglu", 1024, 5000, 64)])
@pytest.mark.parametrize("B", [3, 8, 32])
def test_batched_forward_on_fp8_rows(pi, act, d, ffn, r, B):
    """Batches of 3 or more tokens: the batched predictor (fp16 predictor
    weights, so the same sets as the fp16 layer) and the E4M3 rows on the
    tensor cores (the W_down^T row scale carried by the activation)."""
    spec = LayerSpec(d=d, ffn=ffn, rank=r, act=act, mean_f=0.1)
    t = make_layer(spec, 26, 0)
    layer = pi.Layer.from_dict(to_dev(t), rows="fp8")
    L8 = Q.fp8_layer(stored_oracle(layer, t))
    x = make_tokens(d, B, seed=50 + B)
    y, idx, count = layer.forward(x.cuda())
    torch.cuda.synchronize()
    S = idx[:int(count.item())].cpu().numpy().astype(np.int64)
    h = O.predictor_hidden(L8, x)
    check_union_set(S, O.predictor_logits(L8, h), O.logit_error_bound(L8, x, h, split=True))
    rows = [0, B // 2, B - 1]
    check_y(y.cpu().numpy()[rows], oracle_y_for_valid_set(L8, x[rows], S))
    assert layer.device_status() == 0


def test_fp8_row_access(pi):
    spec = LayerSpec(d=256, ffn=512, rank=16, mean_f=0.2)
    t = to_dev(make_layer(spec, 24, 0))
    layer = pi.Layer.from_dict(t, rows="fp8")
    with pytest.raises(pi.PiError):
        layer.rows_fp8(1)                           # no gate rows in a ReLU layer
    fp16 = pi.Layer.from_dict(t)
    with pytest.raises(pi.PiError):
        fp16.rows_fp8(0)
