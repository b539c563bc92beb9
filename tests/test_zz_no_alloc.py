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
    """A batch of 3 is always refused; d = 16384 at B = 2 needs
    4 * SMs * 2 * 16384 bytes of scratch, refused exactly when that exceeds
    the 16 MiB array (more than 128 SMs), else computed like pi_sparse_ffn."""
    d, ffn = 16384, 512
    t = make_layer(LayerSpec(d=d, ffn=ffn, rank=64, mean_f=0.1), 78)
    layer = pi.Layer.from_dict(to_dev(t))
    x = make_tokens(d, 3, seed=5).cuda()
    idx = torch.arange(ffn, dtype=torch.int32, device="cuda")
    count = torch.tensor([ffn], dtype=torch.int32, device="cuda")
    y = torch.empty(3, d, dtype=torch.float32, device="cuda")
    assert _noalloc(pi, layer, x, idx, count, y) == 2          # batch of 3
    assert b"1 or 2 tokens" in pi.lib.pi_last_error()
    small = make_layer(LayerSpec(d=256, ffn=512, rank=16, mean_f=0.2), 24)
    q8 = pi.Layer.from_dict(to_dev(small), rows="fp8")          # E4M3 rows: fp16 only here
    xs = make_tokens(256, 1, seed=2).cuda()
    assert _noalloc(pi, q8, xs, idx, count, y[:1, :256].contiguous()) == 2
    assert b"fp16 rows" in pi.lib.pi_last_error()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    need = 4 * sms * 2 * d                                      # one split per SM above d = 2048
    st = _noalloc(pi, layer, x[:2], idx, count, y[:2])
    if need > 16 << 20:
        assert st == 2 and b"scratch" in pi.lib.pi_last_error()
    else:
        assert st == 0 and pi.lib.pi_last_error() == b""
        torch.cuda.synchronize()
        check_y(y[:2].cpu().numpy(), layer.sparse_ffn(x[:2], idx, count).cpu().numpy())
    # a successful call leaves no stale error text behind
    x1 = x[:1].contiguous()
    assert _noalloc(pi, layer, x1, idx, count, y[:1]) == 0
    assert pi.lib.pi_last_error() == b""
    torch.cuda.synchronize()


_MEM_PROBE = r"""
import ctypes as C, sys, torch
sys.path.insert(0, sys.argv[1])
import activation_sparse_rank_gb300 as pi
from workload import LayerSpec, make_layer, make_tokens
t = make_layer(LayerSpec(d=1024, ffn=2048, rank=64, mean_f=0.1), 79)
layer = pi.Layer.from_dict({k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in t.items()})
x = make_tokens(1024, 1, seed=3).cuda()
idx = torch.arange(100, dtype=torch.int32, device="cuda")
count = torch.tensor([100], dtype=torch.int32, device="cuda")
y = torch.empty(1, 1024, dtype=torch.float32, device="cuda")
y2 = layer.sparse_ffn(x, idx, count)          # loads the other kernels' modules first
torch.cuda.synchronize()
def call():
    return pi.lib.pi_sparse_ffn_noalloc(layer.handle, C.c_void_p(x.data_ptr()), 1, C.c_void_p(idx.data_ptr()),
                                        C.c_void_p(count.data_ptr()), C.c_void_p(y.data_ptr()),
                                        C.c_void_p(torch.cuda.current_stream().cuda_stream))
f0 = torch.cuda.mem_get_info()[0]
assert call() == 0
torch.cuda.synchronize()
f1 = torch.cuda.mem_get_info()[0]
assert call() == 0
torch.cuda.synchronize()
f2 = torch.cuda.mem_get_info()[0]
print(f0 - f1, f1 - f2)
"""


def test_noalloc_array_is_reserved_at_first_call(tmp_path):
    """In a fresh process with CUDA's default lazy module loading, the fixed
    array's 16 MiB are taken from the GPU at the entry point's first call,
    and a second call takes nothing more."""
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = {k: v for k, v in os.environ.items() if k != "CUDA_MODULE_LOADING"}
    r = subprocess.run([sys.executable, "-c", _MEM_PROBE, root], capture_output=True, text=True,
                       timeout=300, env=env, cwd=root)
    assert r.returncode == 0, r.stdout + r.stderr
    first, second = (int(v) for v in r.stdout.split()[-2:])
    assert first >= 16 << 20, f"first call took {first} bytes"
    assert second == 0, f"second call took {second} bytes"
