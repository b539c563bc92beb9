"""Pins of the CPU oracle to things other than itself (no GPU needed).

Each test fixes part of the oracle against a hand-worked example, a
pure-Python brute force, a library routine for a special case, an invariant
the method's definition forces, or the actual rounding of binary32.
"""
import numpy as np
import pytest
import torch

from oracle import ffn as O
from oracle import brute
from tests.golden import load as load_golden
from workload import LayerSpec, firing_rates, make_layer, make_tokens
from workload.gen import make_exact_layer, make_exact_tokens


def _layer_from_golden(g):
    t = dict(act=g["act"], W_up=np.atleast_2d(g["W_up"]).astype(np.float16),
             W_gate=np.atleast_2d(g["W_gate"]).astype(np.float16) if "W_gate" in g else None,
             b=g["b"].astype(np.float32), W_down=np.atleast_2d(g["W_down"]).astype(np.float16),
             W_p1=np.atleast_2d(g["W_p1"]).astype(np.float16),
             W_p2=np.atleast_2d(g["W_p2"]).astype(np.float16),
             c_p=g["c_p"].astype(np.float32))
    return O.OracleLayer.from_tensors(t), t


@pytest.mark.parametrize("name", ["tiny_relu.txt", "tiny_reglu.txt"])
def test_hand_worked_example(name):
    g = load_golden(name)
    L, _ = _layer_from_golden(g)
    x = g["x"][None, :].astype(np.float16)
    r = O.predicted_forward(L, x)
    np.testing.assert_array_equal(r["l"][0], g["expect_l"])
    np.testing.assert_array_equal(r["S"], g["expect_S"].astype(np.int64))
    np.testing.assert_array_equal(r["y"][0], g["expect_y"])
    m, _ = O.exact_mask(L, x)
    np.testing.assert_array_equal(np.flatnonzero(m[0]), g["expect_exact_S"].astype(np.int64))
    np.testing.assert_array_equal(O.dense_ffn(L, x)[0], g["expect_y_dense"])


def _tiny(act, seed, d=8, ffn=16, r=4):
    spec = LayerSpec(d=d, ffn=ffn, rank=r, act=act, alpha=1.0, mean_f=0.3,
                     w_std=0.3, wp_std=0.5)
    t = make_layer(spec, seed)
    return O.OracleLayer.from_tensors(t), t


@pytest.mark.parametrize("act", ["relu", "reglu"])
@pytest.mark.parametrize("B", [1, 3])
@pytest.mark.parametrize("seed", [1, 2, 3])
def test_brute_force_tiny(act, B, seed):
    L, t = _tiny(act, seed)
    x = make_tokens(L.d, B, seed=100 + seed)
    r = O.predicted_forward(L, x)
    bf = brute.forward({k: (v.numpy() if hasattr(v, "numpy") else v) for k, v in t.items()}, x.numpy())
    np.testing.assert_array_equal(r["mask"], np.array(bf["mask"]))
    np.testing.assert_array_equal(r["S"], np.array(bf["S"], dtype=np.int64))
    np.testing.assert_allclose(r["y"], np.array(bf["y"]), rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("act", ["relu", "reglu"])
def test_dense_is_library_mlp(act):
    """With every neuron in the set the method is the plain FFN, which torch's
    Linear/ReLU modules compute independently."""
    spec = LayerSpec(d=64, ffn=256, rank=16, act=act, mean_f=0.2)
    t = make_layer(spec, 5)
    L = O.OracleLayer.from_tensors(t)
    x = make_tokens(64, 4, seed=9)
    X = x.double()
    gated = torch.nn.Linear(64, 256, bias=True).double()
    with torch.no_grad():
        gated.weight.copy_((t["W_gate"] if act == "reglu" else t["W_up"]).double())
        gated.bias.copy_(t["b"].double())
        down = torch.nn.Linear(256, 64, bias=False).double()
        down.weight.copy_(t["W_down"].double())
        if act == "relu":
            ref = down(torch.relu(gated(X)))
        else:
            up = torch.nn.Linear(64, 256, bias=False).double()
            up.weight.copy_(t["W_up"].double())
            ref = down(torch.relu(gated(X)) * up(X))
        p1 = torch.nn.Linear(64, 16, bias=False).double()
        p1.weight.copy_(t["W_p1"].double())
        p2 = torch.nn.Linear(16, 256, bias=True).double()
        p2.weight.copy_(t["W_p2"].double())
        p2.bias.copy_(t["c_p"].double())
        lref = p2(torch.relu(p1(X)))
    np.testing.assert_allclose(O.dense_ffn(L, x), ref.numpy(), rtol=1e-11, atol=1e-12)
    l = O.predictor_logits(L, O.predictor_hidden(L, x))
    np.testing.assert_allclose(l, lref.numpy(), rtol=1e-11, atol=1e-12)
    # the threshold is the sigmoid > 1/2 rule away from exact ties
    sig = torch.sigmoid(torch.from_numpy(l)).numpy() > 0.5
    far = np.abs(l) > 1e-12
    np.testing.assert_array_equal(O.predicted_mask(l)[far], sig[far])


@pytest.mark.parametrize("act", ["relu", "reglu"])
def test_sparse_equals_dense_under_exact_mask(act):
    """Neurons outside the exact mask have activation exactly 0, so the sparse
    sum over the exact mask is the dense sum, bit for bit in float64."""
    spec = LayerSpec(d=256, ffn=1024, rank=32, act=act, mean_f=0.1)
    L = O.OracleLayer.from_tensors(make_layer(spec, 11))
    x = make_tokens(256, 3, seed=12)
    m, _ = O.exact_mask(L, x)
    S = O.active_union(m)
    assert 0 < S.size < L.ffn
    np.testing.assert_array_equal(O.sparse_ffn(L, x, S), O.dense_ffn(L, x))


def test_neurons_outside_set_contribute_nothing():
    spec = LayerSpec(d=128, ffn=512, rank=16, act="reglu", mean_f=0.1)
    t = make_layer(spec, 13)
    L = O.OracleLayer.from_tensors(t)
    x = make_tokens(128, 2, seed=14)
    S = O.predicted_forward(L, x)["S"]
    y = O.sparse_ffn(L, x, S)
    out = np.setdiff1d(np.arange(L.ffn), S)
    P = O.OracleLayer.from_tensors(t)
    P.W_up = P.W_up.copy(); P.W_gate = P.W_gate.copy(); P.W_down = P.W_down.copy()
    P.W_up[out] = np.float16(np.nan)
    P.W_gate[out] = np.float16(np.inf)
    P.W_down[:, out] = np.float16(np.nan)
    y2 = O.sparse_ffn(P, x, S)
    assert np.isfinite(y2).all()
    np.testing.assert_array_equal(y, y2)


def test_empty_and_full_sets():
    spec = LayerSpec(d=64, ffn=128, rank=8)
    L = O.OracleLayer.from_tensors(make_layer(spec, 15))
    x = make_tokens(64, 2, seed=16)
    assert (O.sparse_ffn(L, x, np.array([], dtype=np.int64)) == 0).all()
    np.testing.assert_array_equal(O.sparse_ffn(L, x, np.arange(128)), O.dense_ffn(L, x))


def test_union_over_batch():
    rng = np.random.default_rng(0)
    mask = rng.random((5, 300)) < 0.1
    S = O.active_union(mask)
    ref = sorted(set(i for b in range(5) for i in range(300) if mask[b, i]))
    assert S.tolist() == ref
    assert O.active_union(mask[2:3]).tolist() == np.flatnonzero(mask[2]).tolist()
    assert O.active_union(np.zeros((3, 10), bool)).size == 0


def test_zero_logit_is_inactive():
    l = np.array([[0.0, -0.0, 1e-300, -1e-300, 2.0]])
    assert O.predicted_mask(l).tolist() == [[False, False, True, False, True]]


def _fp32_sequential(W16, v32, reverse=False, bias=None):
    """Binary32 dot products W v, summed one term at a time, no FMA."""
    W = W16.astype(np.float32)
    acc = np.zeros(W.shape[0], dtype=np.float32)
    ks = range(W.shape[1])
    for k in (reversed(ks) if reverse else ks):
        acc = (acc + (W[:, k] * v32[k]).astype(np.float32)).astype(np.float32)
    if bias is not None:
        acc = (acc + bias.astype(np.float32)).astype(np.float32)
    return acc


@pytest.mark.parametrize("reverse", [False, True])
def test_logit_error_bound_covers_binary32(reverse):
    spec = LayerSpec(d=1024, ffn=2048, rank=64, mean_f=0.1)
    L = O.OracleLayer.from_tensors(make_layer(spec, 17))
    X = make_tokens(1024, 4, seed=18)
    worst = 0.0
    for t in range(4):
        x16 = X[t].numpy()
        h32 = np.maximum(0, _fp32_sequential(L.W_p1, x16.astype(np.float32), reverse))
        l32 = _fp32_sequential(L.W_p2, h32, reverse, bias=L.c_p)
        # a second order: numpy's own float32 matmul
        h32b = np.maximum(0, L.W_p1.astype(np.float32) @ x16.astype(np.float32))
        l32b = L.W_p2.astype(np.float32) @ h32b + L.c_p
        h = O.predictor_hidden(L, X[t:t + 1])
        l = O.predictor_logits(L, h)[0]
        tau = O.logit_error_bound(L, X[t:t + 1], h)[0]
        for cand in (l32, l32b):
            err = np.abs(cand.astype(np.float64) - l)
            assert (err <= tau).all()
            worst = max(worst, float((err / tau).max()))
        # the band is narrow: few decisions are left open
        assert (np.abs(l) <= tau).mean() < 0.02
    assert worst > 1e-5  # worst-case gamma_n is loose, but not beyond this


def test_preact_error_bound_covers_binary32():
    spec = LayerSpec(d=512, ffn=1024, rank=16, mean_f=0.1)
    L = O.OracleLayer.from_tensors(make_layer(spec, 19))
    X = make_tokens(512, 3, seed=20)
    _, z = O.exact_mask(L, X)
    tau = O.preact_error_bound(L, X)
    for t in range(3):
        z32 = _fp32_sequential(L.W_up, X[t].numpy().astype(np.float32), bias=L.b)
        assert (np.abs(z32 - z[t]) <= tau[t]).all()


def test_logit_error_bound_covers_a_cancelling_hidden_layer():
    # h = 2^24 + 1 - 2^24 = 1, but a binary32 sum in index order rounds
    # 2^24 + 1 to 2^24 (ties to even) and returns h = 0; with W_p2 = +-1 and
    # c_p = -+0.5 both logits change sign.  Only the bound's term for the
    # error of h (e = gamma_d * sum |W_p1 x|) covers that.
    f16, f32 = np.float16, np.float32
    L = O.OracleLayer(act="relu", W_up=np.ones((2, 3), f16), W_gate=None, b=np.zeros(2, f32),
                      W_down=np.ones((3, 2), f16), W_p1=np.array([[1024, 1, -1024]], f16),
                      W_p2=np.array([[1], [-1]], f16), c_p=np.array([-0.5, 0.5], f32))
    x = np.array([[16384, 1, 16384]], f16)
    h = O.predictor_hidden(L, x)
    l = O.predictor_logits(L, h)[0]
    assert h.tolist() == [[1.0]] and l.tolist() == [0.5, -0.5]
    h32 = np.maximum(0, _fp32_sequential(L.W_p1, x[0].astype(np.float32)))
    l32 = _fp32_sequential(L.W_p2, h32, bias=L.c_p)
    assert h32.tolist() == [0.0] and l32.tolist() == [-0.5, 0.5]   # both decisions flip
    tau = O.logit_error_bound(L, x, h)[0]
    assert (np.abs(l32 - l) <= tau).all()
    assert O.predicted_mask(l).tolist() == [True, False]


def test_profile_band_counts_only_undecided_pairs():
    # pre-activations exactly 0, 0 and 7 for the token x = (1, 1): the first
    # two are inside the binary32 band (either decision is a correct binary32
    # result), the third is forced; none of them fires in exact arithmetic
    # except the third
    f16, f32 = np.float16, np.float32
    L = O.OracleLayer(act="relu", W_up=np.array([[1, 1], [1, -1], [2, 0]], f16), W_gate=None,
                      b=np.array([-2, 0, 5], f32), W_down=np.ones((2, 3), f16),
                      W_p1=np.ones((1, 2), f16), W_p2=np.ones((3, 1), f16), c_p=None)
    X = np.array([[1, 1], [1, 1], [-1, 2]], f16)      # z = (0, 0, 7), (0, 0, 7), (-1, -3, 3)
    counts, band = O.profile_counts(L, X)
    assert counts.tolist() == [0, 0, 3]
    assert band.tolist() == [2, 2, 0]


def test_preact_error_bound_covers_a_bias_dominated_sum():
    # z = 2^-12 * 2^-13 + 1 = 1 + 2^-25: binary32 rounds the last addition
    # to 1, an error of 2^-25 that only the bound's |b| term covers
    f16, f32 = np.float16, np.float32
    L = O.OracleLayer(act="relu", W_up=np.array([[2.0 ** -12]], f16), W_gate=None,
                      b=np.array([1.0], f32), W_down=np.ones((1, 1), f16),
                      W_p1=np.ones((1, 1), f16), W_p2=np.ones((1, 1), f16), c_p=None)
    x = np.array([[2.0 ** -13]], f16)
    _, z = O.exact_mask(L, x)
    z32 = _fp32_sequential(L.W_up, x[0].astype(np.float32), bias=L.b)
    assert z[0, 0] == 1.0 + 2.0 ** -25 and z32[0] == np.float32(1.0)
    assert abs(float(z32[0]) - z[0, 0]) <= O.preact_error_bound(L, x)[0, 0]


def test_activations_and_sum_follow_the_order_of_s():
    # the operators take S in any order: a[:, k] belongs to neuron S[k] and
    # pairs with W_down[:, S[k]]
    spec = LayerSpec(d=64, ffn=200, rank=8, act="reglu", mean_f=0.3)
    L = O.OracleLayer.from_tensors(make_layer(spec, 31))
    x = make_tokens(64, 2, seed=32).numpy()
    S = np.arange(0, 200, 3)
    perm = np.random.default_rng(5).permutation(S.size)
    a = O.ffn_activations(L, x, S)
    a_p = O.ffn_activations(L, x, S[perm])
    assert np.array_equal(a_p, a[:, perm])
    y = O.ffn_output(L, S, a)
    y_p = O.ffn_output(L, S[perm], a_p)
    assert np.allclose(y_p, y, rtol=1e-12, atol=1e-12 * np.abs(y).max())


def test_firing_rate_construction():
    f, c = firing_rates(4096, 1.0, 0.10, 0.9, seed=3)
    assert abs(f.mean() - 0.10) < 1e-9
    assert f.max() <= 0.9 + 1e-15
    # uncapped neurons follow c * rank^-alpha: f * rank is constant
    order = np.argsort(-f, kind="stable")
    rank = np.arange(1, 4097, dtype=np.float64)
    unc = f[order] < 0.9
    np.testing.assert_allclose(f[order][unc] * rank[unc], c, rtol=1e-12)


def test_generator_fires_at_target_rates():
    """Empirical exact-mask rate over many tokens matches f_i (binomial 5 sigma)."""
    spec = LayerSpec(d=1024, ffn=4096, rank=64, mean_f=0.10)
    t = make_layer(spec, 21)
    L = O.OracleLayer.from_tensors(t)
    T = 4000
    X = make_tokens(1024, T, seed=22)
    counts, _ = O.profile_counts(L, X, chunk=1000)
    f = t["f"].numpy()
    sd = np.sqrt(T * f * (1 - f))
    assert (np.abs(counts - T * f) <= 5 * sd + 1).all()
    assert abs(counts.sum() / (T * 4096) - 0.10) < 0.005


@pytest.mark.parametrize("act", ["relu", "reglu", "swiglu"])
def test_bias_gives_each_neuron_its_target_firing_probability(act):
    # for x ~ N(0, I) the gated pre-activation of neuron i is normal with
    # standard deviation ||W_i|| (the gate's row for gated layers), so it is
    # positive with probability Phi(b_i / ||W_i||), which must be f_i
    from scipy.stats import norm
    spec = LayerSpec(d=256, ffn=1024, rank=16, act=act, mean_f=0.15)
    t = make_layer(spec, 29)
    W = (t["W_gate"] if act != "relu" else t["W_up"]).double().numpy()
    p = norm.cdf(t["b"].double().numpy() / np.linalg.norm(W, axis=1))
    assert np.abs(p - t["f"].numpy()).max() < 1e-6


def test_predictor_logit_moments_match_monte_carlo():
    # mean and variance of W_p2_i . ReLU(W_p1 x) over x ~ N(0, I), which set
    # the calibrated c_p, against 400k sampled tokens (6 standard errors)
    from workload.gen import predictor_logit_moments
    g = np.random.default_rng(41)
    W_p1 = g.normal(0, 0.3, (6, 16)).astype(np.float16)
    W_p2 = g.normal(0, 0.3, (5, 6)).astype(np.float16)
    mu, var = (m.numpy() for m in predictor_logit_moments(torch.from_numpy(W_p1), torch.from_numpy(W_p2)))
    N = 400_000
    x = g.standard_normal((N, 16))
    l0 = np.maximum(0.0, x @ W_p1.astype(np.float64).T) @ W_p2.astype(np.float64).T
    m_hat, v_hat = l0.mean(axis=0), l0.var(axis=0)
    se_m = np.sqrt(v_hat / N)
    se_v = np.sqrt(((l0 - m_hat) ** 4).mean(axis=0) / N)
    assert (np.abs(m_hat - mu) <= 6 * se_m).all()
    assert (np.abs(v_hat - var) <= 6 * se_v).all()


def test_calibrated_predictor_density():
    spec = LayerSpec(d=1024, ffn=4096, rank=64, mean_f=0.10)
    t = make_layer(spec, 23)
    L = O.OracleLayer.from_tensors(t)
    X = make_tokens(1024, 512, seed=24)
    l = O.predictor_logits(L, O.predictor_hidden(L, X))
    dens = O.predicted_mask(l).mean()
    assert 0.08 < dens < 0.12, dens
    # the hot neurons are also the ones predicted most often
    f = t["f"].numpy()
    rate = O.predicted_mask(l).mean(axis=0)
    assert np.corrcoef(rate, f)[0, 1] > 0.9
    # literal predictor (no output bias): logits centre near zero, about half fire
    L.c_p = None
    l0 = O.predictor_logits(L, O.predictor_hidden(L, X))
    assert 0.3 < O.predicted_mask(l0).mean() < 0.7


def test_profile_counts_brute():
    L, t = _tiny("relu", 4, d=8, ffn=16, r=4)
    X = make_tokens(8, 50, seed=25)
    counts, _ = O.profile_counts(L, X, chunk=7)
    Wu, b = t["W_up"].double().numpy(), t["b"].double().numpy()
    ref = [sum(1 for x in X.double().numpy() if sum(Wu[i, j] * x[j] for j in range(8)) + b[i] > 0)
           for i in range(16)]
    assert counts.tolist() == ref


def test_hot_first_order():
    c = np.array([3, 7, 7, 0, 3, 9, 0])
    p = O.hot_first_order(c)
    assert p.tolist() == [5, 1, 2, 0, 4, 3, 6]
    rng = np.random.default_rng(1)
    c = rng.integers(0, 5, 1000)
    p = O.hot_first_order(c)
    assert sorted(p.tolist()) == list(range(1000))
    ref = sorted(range(1000), key=lambda i: (-c[i], i))
    assert p.tolist() == ref


def test_permutation_invariance():
    spec = LayerSpec(d=128, ffn=512, rank=16, act="reglu", mean_f=0.15)
    L = O.OracleLayer.from_tensors(make_layer(spec, 26))
    x = make_tokens(128, 2, seed=27)
    perm = np.random.default_rng(2).permutation(512)
    P = O.permute_layer(L, perm)
    r0, r1 = O.predicted_forward(L, x), O.predicted_forward(P, x)
    assert sorted(perm[r1["S"]].tolist()) == r0["S"].tolist()
    np.testing.assert_allclose(r1["y"], r0["y"], rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("act", ["relu", "reglu"])
def test_exact_arithmetic_mode(act):
    """Integer-grid data: every binary32 partial sum is exact, so a binary32
    evaluation in any order equals float64; exact ties l == 0 occur."""
    t = make_exact_layer(256, 512, 32, act=act, seed=3)
    L = O.OracleLayer.from_tensors(t)
    X = make_exact_tokens(256, 8, seed=4)
    r = O.predicted_forward(L, X)
    assert (r["l"] == 0).any()            # the tie rule is exercised
    # realised magnitude bound: sum of |terms| stays on the 2^-9 grid below 2^24
    a = O.ffn_activations(L, X, r["S"])
    Wd = np.abs(L.W_down[:, r["S"]].astype(np.float64))
    assert ((np.abs(a) @ Wd.T).max() * 512) < 2 ** 24
    for t_ in range(X.shape[0]):
        x32 = X[t_].numpy().astype(np.float32)
        h32 = np.maximum(0, _fp32_sequential(L.W_p1, x32))
        l32 = _fp32_sequential(L.W_p2, h32, bias=L.c_p)
        np.testing.assert_array_equal(l32.astype(np.float64), r["l"][t_])


# --------------------------------------------------------------------------
# SwiGLU (a_i = SiLU(gate) * up over the kept neurons)
# --------------------------------------------------------------------------

def test_silu_closed_forms():
    z = np.array([-50.0, -3.0, -1.0, 0.0, 0.5, 2.0, 40.0])
    s = O.silu(z)
    assert s[3] == 0.0
    assert np.allclose(s - O.silu(-z), z, rtol=0, atol=1e-15)      # SiLU(z) - SiLU(-z) = z
    assert np.allclose(s, z / (1.0 + np.exp(-z)), rtol=1e-15, atol=1e-300)
    assert abs(s[-1] - 40.0) < 1e-15 and abs(s[0]) < 1e-20


def test_swiglu_dense_matches_torch_modules():
    spec = LayerSpec(d=48, ffn=40, rank=8, act="swiglu", mean_f=0.5)
    t = make_layer(spec, 13, 0)
    L = O.OracleLayer.from_tensors(t)
    x = make_tokens(48, 3, seed=5)
    gate = torch.nn.Linear(48, 40, dtype=torch.float64)
    up = torch.nn.Linear(48, 40, bias=False, dtype=torch.float64)
    down = torch.nn.Linear(40, 48, bias=False, dtype=torch.float64)
    with torch.no_grad():
        gate.weight.copy_(t["W_gate"].double()); gate.bias.copy_(t["b"].double())
        up.weight.copy_(t["W_up"].double()); down.weight.copy_(t["W_down"].double())
        ref = down(torch.nn.functional.silu(gate(x.double())) * up(x.double())).numpy()
    assert np.allclose(O.dense_ffn(L, x), ref, rtol=1e-12, atol=1e-12)


def test_swiglu_sparse_sums_split_the_dense_sum_and_match_brute_force():
    spec = LayerSpec(d=16, ffn=24, rank=4, act="swiglu", mean_f=0.5)
    t = make_layer(spec, 17, 0)
    L = O.OracleLayer.from_tensors(t)
    x = make_tokens(16, 2, seed=9)
    r = O.predicted_forward(L, x)
    S = r["S"]
    rest = np.setdiff1d(np.arange(24), S)
    # the pruned neurons' terms are exactly what the sparse sum leaves out
    assert np.allclose(O.sparse_ffn(L, x, S) + O.sparse_ffn(L, x, rest), O.dense_ffn(L, x),
                       rtol=1e-12, atol=1e-14)
    bf = brute.forward({k: (v.numpy() if hasattr(v, "numpy") else v) for k, v in t.items()}, x.numpy())
    assert bf["S"] == list(S)
    assert np.allclose(np.array(bf["y"]), r["y"], rtol=1e-12, atol=1e-14)


def test_fp16_pair_error_bound():
    """The hi/lo fp16 split of binary32 values (the tensor-core form of h)
    stays within fp16_pair_error_bound, on random values over many binades
    and on hand-made values where each term of the bound is the one that
    matters."""
    rng = np.random.default_rng(5)
    v = (rng.standard_normal(200000) * np.exp2(rng.integers(-12, 12, 200000))).astype(np.float32)
    # 2^-6 + 3 * 2^-27: hi = 2^-6, the remainder 0.375 * 2^-24 rounds to lo = 0
    # (fp16 subnormal spacing 2^-24): an error of 3 * 2^-27, above the relative
    # term 2^-22 * 2^-6 = 2^-28; only the 2^-25 term covers it
    sub = np.float32(2.0 ** -6 + 3 * 2.0 ** -27)
    # 1 + 2^-11 + 2^-22 + 2^-23: the remainder needs more bits than fp16 keeps
    rel = np.float32(1 + 2.0 ** -11 + 2.0 ** -22 + 2.0 ** -23)
    v = np.concatenate([v, [sub, -sub, rel, -rel]]).astype(np.float32)
    hi, lo = O.fp16_pair(v)
    err = np.abs(v.astype(np.float64) - hi.astype(np.float64) - lo.astype(np.float64))
    bound = O.fp16_pair_error_bound(v)
    assert (err <= bound).all()
    assert err[-4] == 3 * 2.0 ** -27 and err[-4] > 2.0 ** -22 * float(sub)
    assert err[-2] > 0


def test_logit_error_bound_split_covers_the_tensor_core_form():
    """Logits formed as on tensor cores (h in binary32, split into an fp16
    pair, 2r fp16 products summed in binary32 in two orders) stay within the
    split form of the bound, which is never below the plain one."""
    spec = LayerSpec(d=512, ffn=1024, rank=64, mean_f=0.1)
    L = O.OracleLayer.from_tensors(make_layer(spec, 23))
    X = make_tokens(512, 3, seed=24)
    W2 = L.W_p2.astype(np.float32)
    for t in range(3):
        x16 = X[t].numpy()
        h32 = np.maximum(0, _fp32_sequential(L.W_p1, x16.astype(np.float32))).astype(np.float32)
        hi, lo = O.fp16_pair(h32)
        h = O.predictor_hidden(L, X[t:t + 1])
        l = O.predictor_logits(L, h)[0]
        tau_s = O.logit_error_bound(L, X[t:t + 1], h, split=True)[0]
        assert (tau_s >= O.logit_error_bound(L, X[t:t + 1], h)[0]).all()
        for order in (0, 1):
            acc = np.zeros(L.ffn, np.float32)
            pairs = [(W2[:, k] * hi[k].astype(np.float32), W2[:, k] * lo[k].astype(np.float32))
                     for k in range(L.rank)]
            seq = [p for pr in pairs for p in pr] if order == 0 else [pr[1] for pr in pairs] + [pr[0] for pr in pairs]
            for term in seq:
                acc = (acc + term.astype(np.float32)).astype(np.float32)
            acc = (acc + L.c_p.astype(np.float32)).astype(np.float32)
            assert (np.abs(acc.astype(np.float64) - l) <= tau_s).all()
