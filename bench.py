#!/usr/bin/env python
"""Throughput of the predictor-gated sparse FFN on one GB300 (or N replicas).

Metric: sparse-FFN tokens/s at batch 1, and the effective HBM bandwidth on the
weight bytes actually touched (predictor + active rows) against peak.

A step is one pass of the whole path over one batch of synthetic input: the
256 decode tokens of the OPT-7B-shaped stack (d=4096, ffn=16384, r=256,
32 layers, hot-first neuron order from a 10k-token profile), each token
through all 32 layers in order (predictor, active list, sparse FFN), batch 1.
The step is one CUDA graph launch.  Each step streams about 1.2 GB of distinct
weight rows through a 129 MB L2, so inputs are larger than L2 between steps.

Prints one JSON line (rank 0).  ``--impl reference`` times the float64 CPU
oracle on the host cores instead (the reference arm).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time
from pathlib import Path

import numpy as np
import torch

ROOT = Path(__file__).resolve().parent
sys.path.insert(0, str(ROOT))

from workload import config_by_name, make_layer, make_tokens, sub_seed  # noqa: E402

METRIC = "sparse-FFN tokens/s at batch 1; effective HBM GB/s on touched bytes vs peak"
NOMINAL_HBM_GBS = 8000.0
# neurons active on more than this share of the profiled tokens are "hot": the
# step kernel loads the rows of each slice's leading hot places before its
# predictor has decided
HOT_FRAC = 0.5


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="opt7b_stack")
    ap.add_argument("--layers", type=int, default=0, help="override layer count (debug)")
    ap.add_argument("--tokens", type=int, default=0, help="override tokens per step (debug)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--rows", choices=["fp16", "fp8"], default="fp16",
                    help="storage of the gathered up/gate/down rows (fp8: E4M3 codes, per-row scale)")
    ap.add_argument("--batch", default="1",
                    help="tokens per decode batch (the headline metric is batch 1); a comma-separated "
                         "list measures each batch over the same layers, one line each")
    ap.add_argument("--chained", action="store_true",
                    help="time the chained decode step as the main line (x of layer l+1 = "
                         "fp16(y_l / RMS(y_l)) formed on the device)")
    ap.add_argument("--replicas", type=int, default=0,
                    help="copies of the layer stack, each at its own addresses, run one after "
                         "another (0: enough copies that the weights are at least 4x the L2 "
                         "cache, so that every step reads them from HBM)")
    ap.add_argument("--no-chained-line", action="store_true",
                    help="skip the chained-decode figure reported beside the main line")
    return ap.parse_args()


def measured_peaks():
    p = ROOT / "MEASURED_PEAKS.json"
    if p.exists():
        d = json.loads(p.read_text())
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def bytes_per_active_neuron(d: int, act: str, rows: str = "fp16") -> int:
    """Weight bytes read per active neuron: its up row (+ gate row) and its
    W_down^T row, 2d bytes each (fp8 rows: d code bytes + a 4-byte scale)."""
    per_row = d + 4 if rows == "fp8" else 2 * d
    return per_row * (3 if act in ("reglu", "swiglu") else 2)


def predictor_bytes(d: int, ffn: int, r: int) -> int:
    return 2 * r * d + 2 * ffn * r


# --------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ["clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]

    def __init__(self, device_index: int):
        self.proc = None
        self.err = None
        gid = self._gpu_id(device_index)
        cmd = ["nvidia-smi", f"--id={gid}", "--query-gpu=" + ",".join(self.FIELDS),
               "--format=csv,noheader,nounits", "-lms", "100"]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except Exception as e:  # no nvidia-smi
            self.err = str(e)

    @staticmethod
    def _gpu_id(i: int) -> str:
        p = torch.cuda.get_device_properties(i)
        if all(hasattr(p, a) for a in ("pci_domain_id", "pci_bus_id", "pci_device_id")):
            return f"{p.pci_domain_id:08X}:{p.pci_bus_id:02X}:{p.pci_device_id:02X}.0"
        vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
        if vis:
            return vis.split(",")[i]
        return str(i)

    def stop(self):
        if self.proc is None:
            return {"error": self.err or "nvidia-smi unavailable"}
        time.sleep(0.25)
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        rows = []
        for line in out.strip().splitlines():
            parts = [s.strip() for s in line.split(",")]
            if len(parts) != len(self.FIELDS):
                continue
            rows.append(parts)
        if not rows:
            return {"error": "no samples"}
        sm = [float(r[0]) for r in rows if r[0].replace(".", "").isdigit()]
        mx = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            for n, v in zip(names, r[4:]):
                if v.lower() == "active":
                    reasons.add(n)
        loaded = [s for s in sm if s > 0.5 * max(sm)] if sm else []
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": max(mx) if mx else None,
                "samples": len(rows), "reasons": sorted(reasons)}


# --------------------------------------------------------------------------
def build_stack(cfg, device, n_layers, keep_host_layers, rows="fp16", hot_frac=HOT_FRAC,
                replicas: int = 1):
    """The workload's layers (and, with replicas > 1, that many copies of the
    whole stack one after another, each copy's weights at their own device
    addresses)."""
    import activation_sparse_rank_gb300 as pi
    spec = cfg.layer
    layers, host_layers = [], []
    copies = []
    for l in range(n_layers):
        t = make_layer(spec, cfg.seed, l, device=device)
        perm = None
        n_hot = 0
        if cfg.profile_tokens:
            Xp = make_tokens(spec.d, cfg.profile_tokens, sub_seed(cfg.seed, l, "profile"), device)
            counts = pi.profile_activations(t, Xp).cpu().numpy()
            perm = pi.hot_first_perm(counts)
            # hot: active on more than hot_frac of the profiled tokens
            n_hot = int((counts > hot_frac * cfg.profile_tokens).sum())
            del Xp
        layer = pi.Layer.from_dict(t, perm=perm, rows=rows)
        layer.set_hot_count(n_hot)
        layers.append(layer)
        for _ in range(replicas - 1):
            c = pi.Layer.from_dict(t, perm=perm, rows=rows)
            c.set_hot_count(n_hot)
            copies.append(c)
        if l < keep_host_layers:
            host_layers.append({k: (v.cpu() if isinstance(v, torch.Tensor) else v)
                                for k, v in t.items()})
        del t
    torch.cuda.synchronize()
    if replicas > 1:          # copy r of layer l at position r * n_layers + l
        per = replicas - 1
        layers = layers + [copies[l * per + r] for r in range(per) for l in range(n_layers)]
    return layers, host_layers


def hot_concentration(counts, share: float = 0.8) -> float:
    """Smallest fraction of the neurons whose activation counts add up to
    `share` of all activations (the hot neurons of the pages' power-law
    locality: "a few neurons carry most activations")."""
    c = np.sort(np.asarray(counts, dtype=np.float64))[::-1]
    tot = c.sum()
    if tot <= 0:
        return 0.0
    k = int(np.searchsorted(np.cumsum(c), share * tot - 1e-9)) + 1
    return k / c.size


def profile_concentration(cfg, device, tokens: int = 4096) -> dict:
    """The achieved hot concentration of layer 0 of a workload, from an
    activation profile on the GPU (the configured profile length, else
    `tokens` tokens)."""
    import activation_sparse_rank_gb300 as pi
    spec = cfg.layer
    T = cfg.profile_tokens or tokens
    t = make_layer(spec, cfg.seed, 0, device=device)
    Xp = make_tokens(spec.d, T, sub_seed(cfg.seed, 0, "profile"), device)
    counts = pi.profile_activations(t, Xp).cpu().numpy()
    del t, Xp
    return {"share_of_neurons_carrying_80pct": hot_concentration(counts, 0.8),
            "mean_firing_rate": float(counts.mean() / T), "profile_tokens": T, "layer": 0}


def auto_replicas(cfg, n_layers: int, device=None) -> int:
    """Copies of an n_layers stack whose weights together reach 4x the L2."""
    spec = cfg.layer
    rows = 3 if spec.act in ("reglu", "swiglu") else 2
    per_layer = 2 * spec.d * spec.ffn * rows + predictor_bytes(spec.d, spec.ffn, spec.rank)
    l2 = (torch.cuda.get_device_properties(device).L2_cache_size if device is not None
          else 129 * 1024 * 1024)
    total = per_layer * n_layers
    return max(1, -(-4 * l2 // total)) if total < 4 * l2 else 1


def touched_bytes(cfg, counts: torch.Tensor, rows: str = "fp16") -> int:
    spec = cfg.layer
    T, L = counts.shape
    s = int(counts.sum().item())
    return (T * L * predictor_bytes(spec.d, spec.ffn, spec.rank)
            + s * bytes_per_active_neuron(spec.d, spec.act, rows))


def time_oracle(host_layers, X_host, L_total, seconds: float, min_pairs: int = 4):
    """Float64 oracle on (token, layer) pairs until `seconds` pass; returns
    tokens/s through an L_total-layer stack and a description of the sample."""
    from oracle import ffn as O
    OL = [O.OracleLayer.from_tensors(t) for t in host_layers]
    pairs = 0
    t0 = time.perf_counter()
    tok = 0
    while True:
        for li, L in enumerate(OL):
            O.predicted_forward(L, X_host[tok, li])
            pairs += 1
        tok += 1
        el = time.perf_counter() - t0
        if (el >= seconds and pairs >= min_pairs) or tok >= X_host.shape[0]:
            break
    per_pair = el / pairs
    return 1.0 / (per_pair * L_total), f"{pairs} (token, layer) pairs: tokens 0..{tok - 1} x layers 0..{len(OL) - 1}, {el:.1f} s"


def run_reference(args, cfg):
    """The reference arm: the float64 CPU oracle, timed on the host cores."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    spec = cfg.layer
    n_layers = 2
    Bt = int(str(args.batch).split(",")[0])
    L_total = args.layers or cfg.layers
    host_layers = [{k: (v.cpu() if isinstance(v, torch.Tensor) else v)
                    for k, v in make_layer(spec, cfg.seed, l, device="cpu").items()}
                   for l in range(n_layers)]
    T = max(4, args.steps + args.warmup) * 2
    X = make_tokens(spec.d, T * n_layers * Bt, sub_seed(cfg.seed, 0, "bench_x"), "cpu").view(T, n_layers, Bt, spec.d)
    per_step = max(1.0, min(20.0, 60.0 / max(1, args.steps + args.warmup)))
    from oracle import ffn as O
    OL = [O.OracleLayer.from_tensors(t) for t in host_layers]
    if args.rows == "fp8":                       # the FFN of the E4M3 rows
        from oracle import quant as Q
        OL = [Q.fp8_layer(L) for L in OL]

    def one_step(tok0):
        t0 = time.perf_counter()
        pairs = 0
        tok = tok0
        while True:
            for li, L in enumerate(OL):
                O.predicted_forward(L, X[tok % T, li])
                pairs += 1
            tok += 1
            if time.perf_counter() - t0 >= per_step:
                break
        return time.perf_counter() - t0, pairs, tok

    tok = 0
    for _ in range(args.warmup):
        _, _, tok = one_step(tok)
    tot_t, tot_p = 0.0, 0
    for _ in range(args.steps):
        el, p, tok = one_step(tok)
        tot_t += el
        tot_p += p
    value = Bt / ((tot_t / tot_p) * L_total)
    cores = os.cpu_count()
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1000.0 * tot_t / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(cfg, L_total, args.tokens or cfg.tokens, Bt,
                                  int(os.environ.get("WORLD_SIZE", "1")), args.rows, args.chained,
                                  args.replicas or auto_replicas(cfg, L_total)),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": f"{tot_p} (token, layer) pairs of layers 0..{n_layers - 1}, "
                                   f"{tot_t:.1f} s, batch {Bt}, scaled to a {L_total}-layer stack; numpy "
                                   f"float64 with its default BLAS threads"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def workload_config(cfg, n_layers: int, T: int, Bt: int, world: int, rows: str = "fp16",
                    chained: bool = False, replicas: int = 1) -> dict:
    """The config object both arms print for one workload."""
    spec = cfg.layer
    weights = "fp16" if rows == "fp16" else "fp16 predictor; up/gate/down rows FP8 E4M3 with a per-row fp32 scale"
    return {"workload": cfg.description, "name": cfg.name, "d": spec.d, "ffn": spec.ffn,
            "rank": spec.rank, "layers": n_layers, "tokens_per_step": T * Bt * replicas, "batch": Bt,
            "replicas": replicas,
            "act": spec.act, "weights": weights, "hot_first": bool(cfg.profile_tokens),
            "l2": ("inputs larger than L2: the distinct weight rows of a step exceed the 129 MB L2"
                   if replicas == 1 else
                   f"inputs larger than L2: {replicas} copies of the stack at their own addresses, "
                   "run one after another, hold at least 4x the 129 MB L2"),
            "parallelism": f"replicas{world}",
            "inputs": ("chained: x of layer l+1 = fp16(y_l / RMS(y_l)) on the device" if chained
                       else "independent seeded x ~ N(0, I) per (token, layer); layer l+1 starts "
                            "only after layer l's y is complete")}


def max_over_ranks(value: float, device=None) -> float:
    """Largest value over all ranks (the slowest rank sets a timed region)."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device or "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def kernel_source_hash() -> str:
    """Hash of the persistent step kernel's sources: the stored DRAM counters
    hold only while it matches."""
    h = hashlib.sha256()
    csrc = ROOT / "activation_sparse_rank_gb300" / "csrc"
    for name in ("pi_internal.cuh", "pi_persist.cu"):
        h.update((csrc / name).read_bytes())
    return h.hexdigest()[:16]


def main():
    args = parse()
    cfg = config_by_name(args.config)
    if args.impl == "reference":
        run_reference(args, cfg)
        return

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)

    import activation_sparse_rank_gb300 as pi
    from activation_sparse_rank_gb300.stack import SparseFFNStack

    spec = cfg.layer
    n_layers = args.layers or cfg.layers
    T = args.tokens or cfg.tokens
    batches = [int(b) for b in str(args.batch).split(",")]
    rows = args.rows
    # the CPU baseline times the fp16 oracle; it belongs to the fp16 workload
    want_cpu = (not args.no_cpu_baseline) and rank == 0 and world == 1 and 1 in batches and rows == "fp16"
    t_setup = time.perf_counter()
    R = args.replicas or auto_replicas(cfg, n_layers, device)
    layers, host_layers = build_stack(cfg, device, n_layers, keep_host_layers=2 if want_cpu else 0,
                                      rows=rows, replicas=R)
    NL = len(layers)                      # layers one token passes: R copies of the stack

    def measure(Bt, t_setup):
        stack = SparseFFNStack(layers, tokens=T, B=Bt, chained=args.chained)
        X = make_tokens(spec.d, T * NL * Bt, sub_seed(cfg.seed, 1000 + rank, "bench_x"), device)
        stack.x.copy_(X.view(T, NL, Bt, spec.d))
        del X
        stack.build_graph()
        torch.cuda.synchronize()
        setup_s = time.perf_counter() - t_setup
        cpu_here = want_cpu and Bt == 1

        def barrier():
            if world > 1:
                torch.distributed.barrier()

        s = stack.stream
        for _ in range(max(3, args.warmup)):
            with torch.cuda.stream(s):
                stack.graph.replay()
        s.synchronize()

        clocks = ClockSampler(local)
        evs_step = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
        barrier()
        torch.cuda.synchronize()
        evs_step[0].record(s)
        with torch.cuda.stream(s):
            for k in range(args.steps):
                stack.graph.replay()
                evs_step[k + 1].record(s)
        torch.cuda.synchronize()
        barrier()
        clk = clocks.stop()
        step_ms = [evs_step[k].elapsed_time(evs_step[k + 1]) for k in range(args.steps)]
        ms = max_over_ranks(evs_step[0].elapsed_time(evs_step[-1]) / args.steps, device=device)
        for layer in layers:
            if layer.device_status() != 0:
                raise RuntimeError("device check failed during the timed steps")

        tokens_step = T * Bt * R            # tokens of the n_layers-layer workload per step
        value = tokens_step * world / (ms / 1000.0)
        repeats = {"n": len(step_ms), "median_ms": statistics.median(step_ms), "min_ms": min(step_ms),
                   "max_ms": max(step_ms),
                   "median_tokens_per_s": tokens_step * world / (statistics.median(step_ms) / 1000.0),
                   "max_tokens_per_s": tokens_step * world / (min(step_ms) / 1000.0)}
        tb = touched_bytes(cfg, stack.count, rows)
        mean_S = float(stack.count.double().mean().item())
        eff_gbs = tb / (ms / 1000.0) / 1e9
        peak, peak_kind = measured_peaks()
        gpu_launches = stack.launches_per_step() * args.steps

        # dense comparator: the same kernels over every neuron, 16 tokens (fp16
        # rows only: the standalone operators read fp16 rows)
        dense_tok_s = None
        if rows == "fp16":
            Td = min(16, T)
            dense_g = torch.cuda.CUDAGraph()
            ws = stack.ws
            yd = torch.empty(NL, Bt, spec.d, dtype=torch.float32, device=device)
            with torch.cuda.stream(s):
                for li, layer in enumerate(layers):
                    layer.dense_ref(stack.x[0, li], yd[li], ws=ws, stream=s)
            s.synchronize()
            with torch.cuda.graph(dense_g, stream=s):
                for t in range(Td):
                    for li, layer in enumerate(layers):
                        layer.dense_ref(stack.x[t, li], yd[li], ws=ws, stream=s)
            for _ in range(2):
                dense_g.replay()
            torch.cuda.synchronize()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(s)
            with torch.cuda.stream(s):
                for _ in range(3):
                    dense_g.replay()
            e1.record(s)
            torch.cuda.synchronize()
            dense_tok_s = 3 * Td * Bt * R / (e0.elapsed_time(e1) / 1000.0)

        # dominant kernel (the persistent step kernel, one launch per token)
        # timed inside a captured step with external event-record nodes
        Tr = min(64, T)
        try:
            evs = {t: (torch.cuda.Event(enable_timing=True, external=True),
                       torch.cuda.Event(enable_timing=True, external=True)) for t in range(Tr)}
            how = "external event-record nodes around each launch inside a captured step"
        except TypeError:
            evs = None
            how = None
        if evs is not None:
            for a, b in evs.values():      # materialise the events before capture
                a.record(s); b.record(s)
            s.synchronize()
            g_inst = stack.capture(timing_events=evs, tokens=Tr)
            with torch.cuda.stream(s):
                g_inst.replay()
            s.synchronize()
        else:
            evs = {t: (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for t in range(Tr)}
            with torch.cuda.stream(s):
                for t in range(Tr):
                    layers[0].set_timing_events(*evs[t])
                    stack._token(t, s)
                    layers[0].set_timing_events(None, None)
            s.synchronize()
            how = "events around each launch, eager step"
        k_ms = [evs[t][0].elapsed_time(evs[t][1]) for t in range(Tr)]
        cnt = stack.count[:Tr].cpu().numpy()
        # layers[0]'s timing hook brackets the launch that holds layer 0: the first
        # PI_STACK_LAYERS_PER_LAUNCH layers of a longer stack
        L1 = min(NL, pi.PI_STACK_LAYERS_PER_LAUNCH)
        if Bt <= 2:   # the persistent step: predictor + rows of the launch's layers
            alg_bytes = (Tr * L1 * predictor_bytes(spec.d, spec.ffn, spec.rank)
                         + float(cnt[:, :L1].sum()) * bytes_per_active_neuron(spec.d, spec.act, rows))
            kname = f"k_stack_step (one token through {L1} layers)"
        else:         # tensor-core up + down of layer 0: its active rows
            alg_bytes = float(cnt[:, 0].sum()) * bytes_per_active_neuron(spec.d, spec.act)
            kname = "k_tc_rows<act> + k_tc_down (layer 0, tcgen05)"
        k_avg_ms = sum(k_ms) / len(k_ms)
        achieved = alg_bytes / len(k_ms) / (k_avg_ms / 1e3) / 1e9
        traffic = None
        tfile = ROOT / "profiles" / "stack_step_traffic.json"
        if tfile.exists():
            tj = json.loads(tfile.read_text())
            # counters of this kernel on this workload's layers, per layer
            if tj.get("kernel_source_hash") == kernel_source_hash() and tj.get("config") == cfg.name:
                traffic = tj["bytes_per_layer"] * L1
        if Bt > 2 or rows != "fp16":     # the stored counters are of the fp16 step kernel
            traffic = None
        roofline = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                    "frac": achieved / peak, "traffic": traffic,
                    "kernel": kname,
                    "peak_kind": peak_kind + " (copy bandwidth)",
                    "launches_timed": len(k_ms), "avg_launch_us": k_avg_ms * 1e3,
                    "algorithmic_bytes_per_launch": alg_bytes / len(k_ms),
                    "timing": how}
        if Bt > 2:
            mult = 3 if spec.act in ("reglu", "swiglu") else 2
            flops = 2.0 * Bt * float(cnt[:, 0].sum()) * spec.d * mult / len(k_ms)
            roofline["tensor_tflops"] = flops / (k_avg_ms / 1e3) / 1e12

        # end to end from pinned host buffers through the public API
        xh = torch.empty_like(stack.x, device="cpu").pin_memory()
        xh.copy_(stack.x)
        yh = torch.empty_like(stack.y, device="cpu").pin_memory()
        for _ in range(2):
            stack.run_host(xh, yh, stream=s)
        s.synchronize()
        E = max(3, min(args.steps, 5))
        f0 = torch.cuda.Event(enable_timing=True)
        f1 = torch.cuda.Event(enable_timing=True)
        f0.record(s)
        for _ in range(E):
            stack.run_host(xh, yh, stream=s)
        f1.record(s)
        s.synchronize()
        e2e_ms = f0.elapsed_time(f1) / E
        e2e = {"value": tokens_step * world / (e2e_ms / 1000.0), "unit": "tokens/s",
               "h2d_bytes_per_step": xh.numel() * xh.element_size(),
               "d2h_bytes_per_step": yh.numel() * yh.element_size()}

        # the same step with each layer's input formed from the previous layer's
        # output on the device (a decoder's dependence), beside the main line
        chained_line = None
        if not args.chained and not args.no_chained_line:
            cst = SparseFFNStack(layers, tokens=T, B=Bt, chained=True)
            cst.x[:, 0].copy_(stack.x[:, 0])
            cst.build_graph()
            for _ in range(2):
                with torch.cuda.stream(cst.stream):
                    cst.graph.replay()
            cst.stream.synchronize()
            c0 = torch.cuda.Event(enable_timing=True)
            c1 = torch.cuda.Event(enable_timing=True)
            Kc = max(3, min(args.steps, 5))
            c0.record(cst.stream)
            with torch.cuda.stream(cst.stream):
                for _ in range(Kc):
                    cst.graph.replay()
            c1.record(cst.stream)
            cst.stream.synchronize()
            c_ms = c0.elapsed_time(c1) / Kc
            c_tb = touched_bytes(cfg, cst.count, rows)
            chained_line = {"value": tokens_step * world / (c_ms / 1000.0), "unit": "tokens/s",
                            "ms_per_step": c_ms, "effective_hbm_gbs": c_tb / (c_ms / 1000.0) / 1e9,
                            "mean_active": float(cst.count.double().mean().item()),
                            "what": "x of layer l+1 = fp16(y_l / RMS(y_l)) formed on the device after "
                                    "layer l completes; only layer 0's x is an input"}
            del cst

        # with copies, the same step over one copy (its weights may stay in L2)
        warm = None
        if R > 1:
            st1 = SparseFFNStack(layers[:n_layers], tokens=T, B=Bt)
            st1.x.copy_(stack.x[:, :n_layers])
            st1.build_graph()
            for _ in range(3):
                with torch.cuda.stream(st1.stream):
                    st1.graph.replay()
            st1.stream.synchronize()
            w0 = torch.cuda.Event(enable_timing=True)
            w1 = torch.cuda.Event(enable_timing=True)
            w0.record(st1.stream)
            with torch.cuda.stream(st1.stream):
                for _ in range(5):
                    st1.graph.replay()
            w1.record(st1.stream)
            st1.stream.synchronize()
            warm = {"value": 5 * T * Bt / (w0.elapsed_time(w1) / 1000.0), "unit": "tokens/s",
                    "what": "one copy of the stack, replayed: its weights can stay in L2"}
            del st1
        concentration = profile_concentration(cfg, device)

        cpu = None
        if cpu_here:
            xh_l = stack.x[:, :2].cpu()
            v, sample = time_oracle(host_layers, xh_l, n_layers, args.cpu_seconds)
            cpu = {"value": v, "unit": "tokens/s", "cores": os.cpu_count(), "kind": "oracle",
                   "sample": sample + f"; scaled to a {n_layers}-layer stack; numpy float64, default BLAS threads"}

        if rank == 0:
            line = {
                "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "f32", "data": "synthetic",
                "config": workload_config(cfg, n_layers, T, Bt, world, rows, args.chained, R),
                "effective_hbm_gbs": eff_gbs,
                "effective_frac_of_measured": eff_gbs / peak,
                "effective_frac_of_nominal_8tbs": eff_gbs / (NOMINAL_HBM_GBS),
                "touched_bytes_per_step": tb, "mean_active": mean_S,
                "dense_tokens_per_s": dense_tok_s,
                "speedup_vs_dense": value / world / dense_tok_s if dense_tok_s else None,
                "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
                "chained_decode": chained_line,
                "repeats": repeats, "warm_l2": warm, "hot_concentration": concentration,
                "gpu_launches": gpu_launches, "clocks": clk, "setup_s": setup_s,
            }
            print(json.dumps(line), flush=True)

    for Bt in batches:
        measure(Bt, t_setup)
        t_setup = time.perf_counter()

    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
