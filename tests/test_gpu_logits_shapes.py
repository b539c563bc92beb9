"""The decode step's logits at slice shapes that choose each form of the
staged W_p2 block: on the tensor cores (rank a multiple of 64; 200-neuron
slices, and 300-neuron slices that need more 16-row tiles than the CTA has
warps), and on the ALU where the rank is not a multiple of 64 (r / 8 = 6: two
threads per row, three vectors each; 527-neuron slices: one thread per row
over two passes of the CTA), against the float64 oracle."""
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


@pytest.mark.parametrize("act,d,ffn,r", [
    ("relu", 1024, 30400, 64),    # 200-neuron slices on 152 SMs: 13 row tiles on the tensor cores
    ("relu", 512, 45600, 64),     # 300-neuron slices: 19 row tiles, more than the CTA's 16 warps
    ("reglu", 512, 4096, 48),     # r / 8 = 6: two threads per row, three vectors each
    ("relu", 256, 80000, 16),     # 527-neuron slices: one thread per row, two passes
])
@pytest.mark.parametrize("B", [1, 2])
def test_step_forward(pi, act, d, ffn, r, B):
    n = 2
    spec = LayerSpec(d=d, ffn=ffn, rank=r, act=act, mean_f=0.1)
    ts = [make_layer(spec, 71, l) for l in range(n)]
    layers = [pi.Layer.from_dict(to_dev(t)) for t in ts]
    x = make_tokens(d, n * B, seed=72).view(n, B, d)
    y = torch.empty(n, B, d, dtype=torch.float32, device="cuda")
    idx = torch.full((n, ffn), -1, dtype=torch.int32, device="cuda")
    count = torch.empty(n, dtype=torch.int32, device="cuda")
    pi.stack_forward(layers, x.cuda(), y, idx=idx, count=count)
    torch.cuda.synchronize()
    for l in range(n):
        L = O.permute_layer(O.OracleLayer.from_tensors(ts[l]), layers[l].perm())
        S = idx[l, : int(count[l].item())].cpu().numpy().astype(np.int64)
        res = O.predicted_forward(L, x[l])
        check_union_set(S, res["l"], res["tau"])
        check_y(y[l].cpu().numpy(), oracle_y_for_valid_set(L, x[l], S))
    assert layers[0].device_status() == 0
