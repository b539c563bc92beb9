"""pi_sparse_ffn_noalloc: the sparse FFN for callers that cannot allocate.

Some callers of this library cannot give it a workspace: their device memory
is already owned by a pool of the framework that hosts them, or they only
receive input and output pointers.  This entry point keeps its scratch in a
fixed array inside the library.  Its result must match pi_sparse_ffn (which
uses a caller workspace) within the tolerance of the other parity tests, on
two calls in a row (the array keeps the previous call's contents).

Collected last on purpose, so a run that stops at the first failure has
already run every other test.
"""
import ctypes as C

import numpy as np
import pytest
import torch

from oracle import ffn as O
from tests.gpu_helpers import check_y, stored_oracle, to_dev
from workload import LayerSpec, make_layer, make_tokens

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pi():
    import __graft_entry__
    __graft_entry__.build()
    import activation_sparse_rank_gb300 as pi
    return pi


def _noalloc(pi, layer, x, idx, count, y):
    return pi.lib.pi_sparse_ffn_noalloc(layer.handle, C.c_void_p(x.data_ptr()), x.shape[0],
                                        C.c_void_p(idx.data_ptr()), C.c_void_p(count.data_ptr()),
                                        C.c_void_p(y.data_ptr()),
                                        C.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("d,ffn,r,act,B", [(4096, 16384, 256, "relu", 1), (1024, 4096, 64, "relu", 2),
                                           (8192, 4096, 128, "reglu", 1)])
def test_noalloc_matches_workspace_path(pi, d, ffn, r, act, B):
    t = make_layer(LayerSpec(d=d, ffn=ffn, rank=r, act=act, mean_f=0.1), 77)
    layer = pi.Layer.from_dict(to_dev(t))
    L = stored_oracle(layer, t)
    for call in range(2):
        x = make_tokens(d, B, seed=100 + call).cuda()
        S = O.predicted_forward(L, x.cpu())["S"]
        idx = torch.from_numpy(S.astype(np.int32)).cuda()
        count = torch.tensor([S.size], dtype=torch.int32, device="cuda")
        y_ref = layer.sparse_ffn(x, idx, count)
        y = torch.full((B, d), float("nan"), dtype=torch.float32, device="cuda")
        assert _noalloc(pi, layer, x, idx, count, y) == 0, pi.lib.pi_last_error()
        torch.cuda.synchronize()
        check_y(y.cpu().numpy(), y_ref.cpu().numpy())
        check_y(y.cpu().numpy(), O.sparse_ffn(L, x.cpu(), S))
    assert layer.device_status() == 0


def test_noalloc_rejects_what_does_not_fit(pi):
    t = make_layer(LayerSpec(d=16384, ffn=512, rank=64, mean_f=0.1), 78)
    layer = pi.Layer.from_dict(to_dev(t))
    x = make_tokens(16384, 3, seed=5).cuda()
    idx = torch.arange(512, dtype=torch.int32, device="cuda")
    count = torch.tensor([512], dtype=torch.int32, device="cuda")
    y = torch.empty(3, 16384, dtype=torch.float32, device="cuda")
    assert _noalloc(pi, layer, x, idx, count, y) == 2          # batch of 3
    assert _noalloc(pi, layer, x[:2], idx, count, y) == 2      # 2 x 16384 partials exceed the array
    assert b"scratch" in pi.lib.pi_last_error()
