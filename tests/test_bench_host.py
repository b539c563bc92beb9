"""Host-side pieces of the benchmark that need no GPU: the algorithmic bytes
per unit of work behind the roofline, and the parsing of the clock samples
taken during the timed region."""
import torch

import bench


def test_algorithmic_bytes_per_unit():
    # per layer and token: the predictor's two matrices (2rd + 2 ffn r bytes
    # of fp16) and, per active neuron, its up (+ gate) row and its W_down^T
    # row of 2d bytes each; E4M3 rows are d code bytes plus a 4-byte scale
    d, ffn, r = 4096, 16384, 256
    assert bench.predictor_bytes(d, ffn, r) == 2 * 256 * 4096 + 2 * 16384 * 256
    assert bench.bytes_per_active_neuron(d, "relu") == 2 * 8192
    assert bench.bytes_per_active_neuron(d, "reglu") == 3 * 8192
    assert bench.bytes_per_active_neuron(d, "swiglu") == 3 * 8192
    assert bench.bytes_per_active_neuron(d, "relu", "fp8") == 2 * 4100
    assert bench.bytes_per_active_neuron(d, "swiglu", "fp8") == 3 * 4100

    class Cfg:
        class layer:
            pass
    Cfg.layer.d, Cfg.layer.ffn, Cfg.layer.rank, Cfg.layer.act = d, ffn, r, "relu"
    counts = torch.tensor([[10, 20, 30], [40, 50, 60]])          # [tokens, layers]
    assert bench.touched_bytes(Cfg, counts) == 6 * bench.predictor_bytes(d, ffn, r) + 210 * 16384


class _FakeSmi:
    def __init__(self, out):
        self.out = out

    def terminate(self):
        pass

    def communicate(self, timeout=None):
        return self.out, ""


def _sampler(out):
    s = object.__new__(bench.ClockSampler)
    s.proc, s.err = _FakeSmi(out), None
    return s


def test_clock_samples_are_summarised():
    rows = [
        "345, 2070, 180.1, 0x0, Not Active, Not Active, Not Active, Not Active",   # idle, before the load
        "2070, 2070, 900.5, 0x0, Not Active, Not Active, Not Active, Not Active",
        "1995, 2070, 1390.0, 0x4, Not Active, Not Active, Not Active, Active",
        "2040, 2070, 1200.0, 0x0, Not Active, Not Active, Not Active, Not Active",
        "garbled line",
    ]
    c = _sampler("\n".join(rows) + "\n").stop()
    assert c["samples"] == 4
    assert c["sm_mhz"] == 2040.0            # median of the loaded samples (idle one left out)
    assert c["sm_max_mhz"] == 2070.0
    assert c["reasons"] == ["sw_power_cap"]


def test_throttle_reasons_are_reported():
    rows = ["1500, 2070, 1400.0, 0x48, Active, Not Active, Active, Not Active"] * 3
    c = _sampler("\n".join(rows)).stop()
    assert c["reasons"] == ["hw_slowdown", "sw_thermal_slowdown"]
    assert _sampler("").stop() == {"error": "no samples"}


def test_hot_concentration():
    import bench
    assert bench.hot_concentration([10, 0, 0, 0]) == 0.25        # one neuron carries everything
    assert bench.hot_concentration([1] * 10) == 0.8               # uniform: 80% of the neurons
    assert abs(bench.hot_concentration([1, 8, 1]) - 1 / 3) < 1e-12
    assert bench.hot_concentration([0, 0]) == 0.0


def test_auto_replicas_only_for_stacks_that_fit_in_l2():
    import bench
    from workload import config_by_name
    l2 = 129 * 1024 * 1024
    c1 = config_by_name("opt_layer_d1024")
    per_layer = 2 * 1024 * 4096 * 2 + bench.predictor_bytes(1024, 4096, 64)
    R = bench.auto_replicas(c1, 1)
    assert R * per_layer >= 4 * l2 > (R - 1) * per_layer
    assert bench.auto_replicas(config_by_name("opt7b_stack"), 32) == 1
