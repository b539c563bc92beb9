"""Parity of the multi-layer decode step (pi_stack_forward, persistent kernel)
and of the full-size workloads, against the float64 CPU oracle."""
import numpy as np
import pytest
import torch

from oracle import ffn as O
from tests.gpu_helpers import check_union_set, check_y, oracle_y_for_valid_set, to_dev
from workload import CONFIGS, LayerSpec, config_by_name, make_layer, make_tokens, sub_seed

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pi():
    import __graft_entry__
    __graft_entry__.build()
    import activation_sparse_rank_gb300 as pi
    return pi


def _stack(pi, spec, n, seed, perms=None):
    ts = [make_layer(spec, seed, l) for l in range(n)]
    layers = [pi.Layer.from_dict(to_dev(t), perm=None if perms is None else perms[l])
              for l, t in enumerate(ts)]
    return ts, layers


def _check_layer(t, x, y, S, perm=None):
    L = O.OracleLayer.from_tensors(t)
    if perm is not None:
        L = O.permute_layer(L, perm)
    x2 = np.atleast_2d(np.asarray(x))
    if x2.shape[0] > 2:       # batched path: h enters the logits as an fp16 pair
        h = O.predictor_hidden(L, x2)
        band = check_union_set(S, O.predictor_logits(L, h), O.logit_error_bound(L, x2, h, split=True))
    else:
        r = O.predicted_forward(L, x)
        band = check_union_set(S, r["l"], r["tau"])
    check_y(y, oracle_y_for_valid_set(L, x, S))
    return band


@pytest.mark.parametrize("act,d,ffn,r", [("relu", 1024, 4096, 64), ("reglu", 2048, 3000, 40),
                                         ("relu", 12288, 2000, 128)])
@pytest.mark.parametrize("B", [1, 2, 3])
def test_stack_forward(pi, act, d, ffn, r, B):
    n = 3
    spec = LayerSpec(d=d, ffn=ffn, rank=r, act=act, mean_f=0.1)
    ts, layers = _stack(pi, spec, n, seed=d + ffn)
    x = make_tokens(d, n * B, seed=3).view(n, B, d)
    y = torch.empty(n, B, d, dtype=torch.float32, device="cuda")
    idx = torch.full((n, ffn), -1, dtype=torch.int32, device="cuda")
    count = torch.empty(n, dtype=torch.int32, device="cuda")
    pi.stack_forward(layers, x.cuda(), y, idx=idx, count=count)
    y2 = torch.empty_like(y)
    pi.stack_forward(layers, x.cuda(), y2, idx=idx, count=count)
    torch.cuda.synchronize()
    assert torch.equal(y, y2)
    for l in range(n):
        c = int(count[l].item())
        S = idx[l, :c].cpu().numpy().astype(np.int64)
        _check_layer(ts[l], x[l], y[l].cpu().numpy(), S, perm=layers[l].perm())
    assert layers[0].device_status() == 0


def test_long_stack_spans_launches(pi):
    """More layers than one persistent launch holds."""
    n, d, ffn, r = 70, 256, 512, 16
    spec = LayerSpec(d=d, ffn=ffn, rank=r, mean_f=0.15)
    ts, layers = _stack(pi, spec, n, seed=5)
    x = make_tokens(d, n, seed=6).view(n, 1, d)
    y = torch.empty(n, 1, d, dtype=torch.float32, device="cuda")
    idx = torch.empty((n, ffn), dtype=torch.int32, device="cuda")
    count = torch.empty(n, dtype=torch.int32, device="cuda")
    pi.stack_forward(layers, x.cuda(), y, idx=idx, count=count)
    torch.cuda.synchronize()
    for l in range(n):
        c = int(count[l].item())
        _check_layer(ts[l], x[l], y[l].cpu().numpy(), idx[l, :c].cpu().numpy().astype(np.int64),
                     perm=layers[l].perm())
    assert layers[0].device_status() == 0


def test_graph_replay_matches_eager(pi):
    from activation_sparse_rank_gb300.stack import SparseFFNStack
    spec = LayerSpec(d=1024, ffn=4096, rank=64, mean_f=0.1)
    ts, layers = _stack(pi, spec, 4, seed=8)
    st = SparseFFNStack(layers, tokens=5, B=1)
    st.x.copy_(make_tokens(1024, 20, seed=9).view(5, 4, 1, 1024).cuda())
    st.enqueue(stream=torch.cuda.current_stream())
    torch.cuda.synchronize()
    y_eager = st.y.clone()
    st.y.zero_()
    st.build_graph()
    st.replay()
    torch.cuda.synchronize()
    assert torch.equal(st.y, y_eager)
    xh = st.x.cpu().pin_memory()
    yh = torch.empty(st.y.shape, dtype=torch.float32).pin_memory()
    st.run_host(xh, yh)
    torch.cuda.synchronize()
    assert torch.equal(yh, y_eager.cpu())


def test_bench_configuration_sampled(pi):
    """The OPT-7B-shaped stack exactly as the benchmark builds and times it
    (32 layers, hot-first order from a 10k-token profile, graph replay of the
    persistent step), checked on sampled (token, layer) pairs."""
    import bench
    from activation_sparse_rank_gb300.stack import SparseFFNStack
    cfg = config_by_name("opt7b_stack")
    spec = cfg.layer
    dev = torch.device("cuda")
    check_layers = [0, 13, 31]
    layers, _ = bench.build_stack(cfg, dev, cfg.layers, keep_host_layers=0)
    T = 3
    st = SparseFFNStack(layers, tokens=T, B=1, want_idx=True)
    X = make_tokens(spec.d, T * cfg.layers, sub_seed(cfg.seed, 1000, "bench_x"), dev)
    st.x.copy_(X.view(T, cfg.layers, 1, spec.d))
    st.build_graph()
    st.replay()
    torch.cuda.synchronize()
    assert layers[0].device_status() == 0
    for l in check_layers:
        t = make_layer(spec, cfg.seed, l, device=dev)
        perm = layers[l].perm()
        t = {k: (v.cpu() if isinstance(v, torch.Tensor) else v) for k, v in t.items()}
        tok = T - 1                     # the active lists hold the last token's sets
        c = int(st.count[tok, l].item())
        S = st.idx[l, :c].cpu().numpy().astype(np.int64)
        _check_layer(t, st.x[tok, l].cpu(), st.y[tok, l].cpu().numpy(), S, perm=perm)
        # profile order: hot-first permutation is a permutation sorted by the GPU profile
        assert sorted(perm.tolist()) == list(range(spec.ffn))


@pytest.mark.parametrize("name", ["llama2_70b_reglu", "falcon40b_stack", "opt175b_stack"])
def test_full_size_layer(pi, name):
    """One layer at the full per-layer size of each larger workload, batch 1
    through the persistent step, plus the workload's larger batches and its
    prompt pass (128 tokens at once for the OPT-175B shape: the low-sparsity
    union, several hundred 128-row tiles) through the batched path."""
    cfg = config_by_name(name)
    spec = cfg.layer
    dev = torch.device("cuda")
    t = make_layer(spec, cfg.seed, 0, device=dev)
    layer = pi.Layer.from_dict(t)
    th = {k: (v.cpu() if isinstance(v, torch.Tensor) else v) for k, v in t.items()}
    del t
    L = O.permute_layer(O.OracleLayer.from_tensors(th), layer.perm())
    batches = (1,) + tuple(b for b in cfg.batches if b > 1) + ((cfg.prompt,) if cfg.prompt else ())
    for B in sorted(set(batches)):
        x = make_tokens(spec.d, B, seed=sub_seed(cfg.seed, B, "full_size_x"))
        y, idx, count = layer.forward(x.to(dev))
        torch.cuda.synchronize()
        S = idx[:int(count.item())].cpu().numpy().astype(np.int64)
        h = O.predictor_hidden(L, x)
        check_union_set(S, O.predictor_logits(L, h), O.logit_error_bound(L, x, h, split=B > 2))
        rows = [0, B // 2, B - 1] if B > 2 else list(range(B))
        y_ref = O.sparse_ffn(L, x[rows], S)
        check_y(y.cpu().numpy()[rows], y_ref)
        if B == cfg.prompt:
            assert S.size > 0.9 * spec.ffn      # the prompt's union is nearly dense
    assert layer.device_status() == 0


@pytest.mark.parametrize("name", ["opt_layer_d1024", "opt7b_stack", "llama2_70b_reglu",
                                  "llama2_70b_swiglu", "falcon40b_stack", "opt175b_stack"])
def test_full_size_layer_literal_predictor(pi, name):
    """The predictor exactly as the pages state it (no output bias: c_p = 0,
    so about half of the neurons are predicted active), one full-size layer
    of each workload, batch 1 (persistent step) and batch 8 (batched path)."""
    cfg = config_by_name(name)
    spec = cfg.layer
    dev = torch.device("cuda")
    t = make_layer(spec, cfg.seed, 0, device=dev)
    t["c_p"] = None
    layer = pi.Layer.from_dict(t)
    th = {k: (v.cpu() if isinstance(v, torch.Tensor) else v) for k, v in t.items()}
    del t
    L = O.permute_layer(O.OracleLayer.from_tensors(th), layer.perm())
    assert L.c_p is None
    for B in (1, 8):
        x = make_tokens(spec.d, B, seed=sub_seed(cfg.seed, B, "literal_x"))
        y, idx, count = layer.forward(x.to(dev))
        torch.cuda.synchronize()
        S = idx[:int(count.item())].cpu().numpy().astype(np.int64)
        h = O.predictor_hidden(L, x)
        check_union_set(S, O.predictor_logits(L, h), O.logit_error_bound(L, x, h, split=B > 2))
        if B == 1:
            assert 0.35 * spec.ffn < S.size < 0.65 * spec.ffn     # symmetric logits: about half
        rows = [0, B - 1]
        check_y(y.cpu().numpy()[rows], O.sparse_ffn(L, x[rows], S))
    assert layer.device_status() == 0


def test_bench_configuration_all_layers_several_tokens(pi):
    """The OPT-7B-shaped stack as the benchmark builds it (32 layers,
    hot-first order from a 10k-token profile, one persistent launch per
    token): four tokens, every layer's active list and output against the
    oracle."""
    import bench
    cfg = config_by_name("opt7b_stack")
    spec = cfg.layer
    dev = torch.device("cuda")
    layers, _ = bench.build_stack(cfg, dev, cfg.layers, keep_host_layers=0)
    T, Lc = 4, cfg.layers
    X = make_tokens(spec.d, T * Lc, sub_seed(cfg.seed, 1000, "bench_x"), dev).view(T, Lc, 1, spec.d)
    ws = layers[0].workspace(1)
    ys = torch.empty(T, Lc, 1, spec.d, dtype=torch.float32, device=dev)
    idx = torch.full((T, Lc, spec.ffn), -1, dtype=torch.int32, device=dev)
    cnt = torch.empty(T, Lc, dtype=torch.int32, device=dev)
    for tok in range(T):
        pi.stack_forward(layers, X[tok].contiguous(), ys[tok], idx=idx[tok], count=cnt[tok], ws=ws)
    torch.cuda.synchronize()
    assert layers[0].device_status() == 0
    Xh, Yh, Ih, Ch = X.cpu(), ys.cpu().numpy(), idx.cpu().numpy(), cnt.cpu().numpy()
    for l in range(Lc):
        t = make_layer(spec, cfg.seed, l, device=dev)
        th = {k: (v.cpu() if isinstance(v, torch.Tensor) else v) for k, v in t.items()}
        del t
        L = O.permute_layer(O.OracleLayer.from_tensors(th), layers[l].perm())
        for tok in range(T):
            S = Ih[tok, l, :Ch[tok, l]].astype(np.int64)
            r = O.predicted_forward(L, Xh[tok, l])
            check_union_set(S, r["l"], r["tau"])
            check_y(Yh[tok, l], oracle_y_for_valid_set(L, Xh[tok, l], S))


def test_hot_hint_changes_no_result(pi):
    """The hot-neuron hint only moves data earlier: outputs are bitwise equal."""
    spec = LayerSpec(d=2048, ffn=8192, rank=128, mean_f=0.1)
    ts, layers = _stack(pi, spec, 3, seed=31)
    x = make_tokens(2048, 3, seed=32).view(3, 1, 2048).cuda()
    y0 = torch.empty(3, 1, 2048, dtype=torch.float32, device="cuda")
    y1 = torch.empty_like(y0)
    idx = torch.empty(3, 8192, dtype=torch.int32, device="cuda")
    cnt0 = torch.empty(3, dtype=torch.int32, device="cuda")
    cnt1 = torch.empty_like(cnt0)
    pi.stack_forward(layers, x, y0, idx=idx, count=cnt0)
    for l in layers:
        l.set_hot_count(3000)
    pi.stack_forward(layers, x, y1, idx=idx, count=cnt1)
    torch.cuda.synchronize()
    assert torch.equal(y0, y1) and torch.equal(cnt0, cnt1)
    with pytest.raises(pi.PiError):
        layers[0].set_hot_count(8193)


def _chained_x_ref(y_prev) -> np.ndarray:
    """The chained input of the next layer from y [B, d]: y / RMS(y) per token,
    RMS(v) = sqrt(mean(v^2) + 1e-12), in float64 (the GPU rounds its binary32
    result to fp16, so the two agree within one fp16 step)."""
    y = np.asarray(y_prev, dtype=np.float64)
    return y / np.sqrt((y * y).mean(axis=-1, keepdims=True) + 1e-12)


def _check_fp16_within_one_step(x_gpu, ref):
    ref16 = ref.astype(np.float16)
    step = np.spacing(np.abs(ref16)).astype(np.float64)
    diff = np.abs(np.asarray(x_gpu, np.float64) - ref16.astype(np.float64))
    assert (diff <= step).all(), f"chained input off by {float((diff / step).max()):.2f} fp16 steps"


@pytest.mark.parametrize("act,d,ffn,r,B,n", [("relu", 1024, 4096, 64, 1, 5),
                                             ("reglu", 2048, 3000, 40, 2, 4),
                                             ("relu", 4096, 6000, 256, 1, 35),
                                             ("relu", 1024, 2048, 64, 3, 4)])
def test_chained_stack(pi, act, d, ffn, r, B, n):
    """Decode chain: layer l >= 1 takes fp16(y_{l-1} / RMS(y_{l-1})), formed on
    the device (across launch boundaries too: 35 layers span two launches).
    Every checked layer is compared with the oracle on the input the GPU used."""
    spec = LayerSpec(d=d, ffn=ffn, rank=r, act=act, mean_f=0.1)
    ts, layers = _stack(pi, spec, n, seed=d + 7 * ffn + B)
    for layer in layers:
        layer.set_hot_count(ffn // 5)
    x = torch.zeros(n, B, d, dtype=torch.float16, device="cuda")
    x[0] = make_tokens(d, B, seed=41 + B).cuda()
    x_first = x[0].clone()
    y = torch.empty(n, B, d, dtype=torch.float32, device="cuda")
    idx = torch.full((n, ffn), -1, dtype=torch.int32, device="cuda")
    count = torch.empty(n, dtype=torch.int32, device="cuda")
    pi.stack_forward(layers, x, y, idx=idx, count=count, chained=True)
    x2 = torch.zeros_like(x)
    x2[0] = x_first
    y2 = torch.empty_like(y)
    pi.stack_forward(layers, x2, y2, idx=idx.clone(), count=count.clone(), chained=True)
    torch.cuda.synchronize()
    assert torch.equal(x[0], x_first), "the chained step must not overwrite x[0]"
    assert torch.equal(y, y2) and torch.equal(x, x2), "chained step not bitwise reproducible"
    xc, yc = x.cpu(), y.cpu().numpy()
    for l in range(1, n):
        _check_fp16_within_one_step(xc[l].numpy(), _chained_x_ref(yc[l - 1]))
    check = list(range(n)) if n <= 6 else [0, 1, 17, 31, 32, 34]
    for l in check:
        c = int(count[l].item())
        S = idx[l, :c].cpu().numpy().astype(np.int64)
        _check_layer(ts[l], xc[l], yc[l], S, perm=layers[l].perm())
    assert layers[0].device_status() == 0


@pytest.mark.parametrize("act,d,ffn,r,B", [("relu", 4096, 8192, 128, 1), ("relu", 4096, 8192, 128, 2),
                                           ("reglu", 2048, 6000, 64, 1), ("relu", 8192, 4096, 64, 1)])
def test_dense_layer_many_windows(pi, act, d, ffn, r, B):
    """About 60% of the neurons active: every CTA's list spans several row
    windows, including the windows' shared-memory extension slots."""
    n = 2
    spec = LayerSpec(d=d, ffn=ffn, rank=r, act=act, mean_f=0.6)
    ts, layers = _stack(pi, spec, n, seed=d + ffn + 3 * B)
    for layer in layers:
        layer.set_hot_count(ffn // 3)
    x = make_tokens(d, n * B, seed=77 + B).view(n, B, d)
    y = torch.empty(n, B, d, dtype=torch.float32, device="cuda")
    idx = torch.full((n, ffn), -1, dtype=torch.int32, device="cuda")
    count = torch.empty(n, dtype=torch.int32, device="cuda")
    pi.stack_forward(layers, x.cuda(), y, idx=idx, count=count)
    torch.cuda.synchronize()
    assert int(count.min().item()) > ffn // 3
    for l in range(n):
        c = int(count[l].item())
        _check_layer(ts[l], x[l], y[l].cpu().numpy(), idx[l, :c].cpu().numpy().astype(np.int64),
                     perm=layers[l].perm())
    assert layers[0].device_status() == 0
