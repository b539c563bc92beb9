"""FP8 (E4M3) row layers on the GPU against the float64 oracle: the stored
codes and scales byte for byte, and the decode step (pi_layer_forward /
pi_stack_forward at 1 and 2 tokens) against the FFN of the dequantised rows."""
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


def test_fp8_layers_reject_the_fp16_only_entry_points(pi):
    spec = LayerSpec(d=256, ffn=512, rank=16, mean_f=0.2)
    t = to_dev(make_layer(spec, 24, 0))
    layer = pi.Layer.from_dict(t, rows="fp8")
    x = make_tokens(256, 3, seed=2).cuda()
    y = torch.empty(3, 256, dtype=torch.float32, device="cuda")
    idx = torch.arange(512, dtype=torch.int32, device="cuda")
    count = torch.tensor([512], dtype=torch.int32, device="cuda")
    for call in (lambda: layer.sparse_ffn(x[:1], idx, count, y[:1]),
                 lambda: layer.dense_ref(x[:1], y[:1]),
                 lambda: layer.forward(x, idx=torch.empty(512, dtype=torch.int32, device="cuda"),
                                       count=torch.empty(1, dtype=torch.int32, device="cuda"), y=y)):
        with pytest.raises(pi.PiError) as e:
            call()
        assert e.value.status == 2                  # PI_ERR_UNSUPPORTED
    with pytest.raises(pi.PiError):
        layer.rows_fp8(1)                           # no gate rows in a ReLU layer
    fp16 = pi.Layer.from_dict(t)
    with pytest.raises(pi.PiError):
        fp16.rows_fp8(0)
