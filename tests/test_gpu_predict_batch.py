"""Parity of the batched predictor (3 <= B <= 32 tokens: hidden layer, logits,
union over the batch and the ascending list in one cooperative launch)
against the float64 oracle.  The union set is checked decision by decision
within the binary32 bound of the fp16-pair form of h, the layer output over
the returned set element by element, and two runs must agree bitwise."""
import numpy as np
import pytest
import torch

from oracle import ffn as O
from tests.gpu_helpers import check_union_set, check_y, oracle_y_for_valid_set, to_dev
from workload import LayerSpec, make_layer, make_tokens

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pi():
    import __graft_entry__
    __graft_entry__.build()
    import activation_sparse_rank_gb300 as pi
    return pi


# (act, d, ffn, r): a 1024-wide layer; d = 1056 (K chunks of an odd number of
# 32-element blocks; the FFN itself then runs off the tensor cores); fewer
# neurons than SMs (empty slices); a gated layer; the OPT-7B shape; 300-neuron
# slices (19 row tiles of 16 for 16 warps) with r = 192
SHAPES = [("relu", 1024, 4096, 64), ("relu", 1056, 100, 64), ("reglu", 2048, 3000, 128),
          ("relu", 4096, 16384, 256), ("relu", 512, 45600, 192)]


@pytest.mark.parametrize("act,d,ffn,r", SHAPES)
@pytest.mark.parametrize("B", [3, 5, 8, 9, 16, 17, 32])
def test_batched_predictor(pi, act, d, ffn, r, B):
    spec = LayerSpec(d=d, ffn=ffn, rank=r, act=act, mean_f=0.1)
    t = make_layer(spec, 500 + d + B, 0)
    layer = pi.Layer.from_dict(to_dev(t))
    L = O.permute_layer(O.OracleLayer.from_tensors(t), layer.perm())
    x = make_tokens(d, B, seed=900 + B)
    y, idx, count = layer.forward(x.cuda())
    y2, idx2, count2 = layer.forward(x.cuda())
    torch.cuda.synchronize()
    c = int(count.item())
    assert int(count2.item()) == c
    assert torch.equal(idx[:c], idx2[:c]) and torch.equal(y, y2)
    S = idx[:c].cpu().numpy().astype(np.int64)
    h = O.predictor_hidden(L, x)
    check_union_set(S, O.predictor_logits(L, h), O.logit_error_bound(L, x, h, split=True))
    rows = list(range(B)) if B <= 9 else [0, 1, B // 2, B - 1]
    check_y(y.cpu().numpy()[rows], oracle_y_for_valid_set(L, x[rows], S))
    assert layer.device_status() == 0


@pytest.mark.parametrize("B", [3, 32])
def test_batched_predictor_literal_mode(pi, B):
    """No output bias (c_p absent): the threshold is l > 0 on W_p2 h alone."""
    spec = LayerSpec(d=2048, ffn=6000, rank=128, mean_f=0.1)
    t = make_layer(spec, 77, 0)
    t["c_p"] = None
    layer = pi.Layer.from_dict(to_dev(t))
    L = O.permute_layer(O.OracleLayer.from_tensors(t), layer.perm())
    x = make_tokens(2048, B, seed=78)
    y, idx, count = layer.forward(x.cuda())
    torch.cuda.synchronize()
    S = idx[:int(count.item())].cpu().numpy().astype(np.int64)
    h = O.predictor_hidden(L, x)
    check_union_set(S, O.predictor_logits(L, h), O.logit_error_bound(L, x, h, split=True))
    assert S.size > 0.5 * spec.ffn            # a union of about-half sets
    check_y(y.cpu().numpy()[[0, B - 1]], oracle_y_for_valid_set(L, x[[0, B - 1]], S))
    assert layer.device_status() == 0


def test_batched_predictor_in_a_stack(pi):
    """Several layers of 8 tokens through pi_stack_forward: the predictor's
    workspace (partial sums, counts, barrier counter) is reused layer after
    layer."""
    n, B = 4, 8
    spec = LayerSpec(d=1024, ffn=4096, rank=64, mean_f=0.1)
    ts = [make_layer(spec, 31, l) for l in range(n)]
    layers = [pi.Layer.from_dict(to_dev(t)) for t in ts]
    x = make_tokens(1024, n * B, seed=32).view(n, B, 1024)
    y = torch.empty(n, B, 1024, dtype=torch.float32, device="cuda")
    idx = torch.full((n, spec.ffn), -1, dtype=torch.int32, device="cuda")
    count = torch.empty(n, dtype=torch.int32, device="cuda")
    pi.stack_forward(layers, x.cuda(), y, idx=idx, count=count)
    torch.cuda.synchronize()
    for l in range(n):
        L = O.permute_layer(O.OracleLayer.from_tensors(ts[l]), layers[l].perm())
        S = idx[l, :int(count[l].item())].cpu().numpy().astype(np.int64)
        h = O.predictor_hidden(L, x[l])
        check_union_set(S, O.predictor_logits(L, h), O.logit_error_bound(L, x[l], h, split=True))
        check_y(y[l].cpu().numpy(), oracle_y_for_valid_set(L, x[l], S))
    assert layers[0].device_status() == 0
