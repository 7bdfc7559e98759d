"""Throughput of the offloading-aware MoE layer forward on GB300.

One step = one whole layer forward (router + prefetch router + delta_hat,
miss handling, permutation, grouped SwiGLU experts + shared experts, LoRE,
combine) over one batch of synthetic tokens, through the library's C ABI.

Default workload: the DeepSeek-V2-Lite-shaped layer (hidden 2048, 64 routed
experts top-6, 2 shared experts, intermediate 1408, LoRE rank 16, 24 of 64
experts resident by the batch prefetch set, HYBRID miss policy) decoding
8 tokens per step.  Weights stream from HBM: the timed steps rotate over
several copies of the layer's weights at distinct addresses, so the expert
bytes one step reads are evicted from L2 (129 MB) before they are read again.

Other workloads (--workload): the Granite, Mixtral (dense and FloE 10 %) and
Qwen2-57B shapes, and dsv2lite-cache-decode-T1: one-token decode steps over a
persistent expert cache (capacity 24, heat decay 0.99) that moe_cache_update
refreshes every step; its line adds the cache's hit rate and admitted experts.
dsv2lite-lookahead-decode-T8: every 8-token step also runs SPICE's
confidence-aware look-ahead over the next 4 layers of a synthetic stack
(moe_prefetch_depth, tau 0.3, d_min 1); its line adds the depth histogram, the
look-ahead call's time and how many of the next layer's routed slots the
prediction covered.

Usage:  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
        [--workload NAME]
Multi-GPU (torchrun): each rank runs an independent replica on its own
tokens (weak scaling, no data-path collective); rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from workloads import CONFIGS, make_lookahead_routers, make_tokens, make_weights  # noqa: E402

# name -> (layer config, tokens per step, phase[, FloE keep fraction])
WORKLOADS = {
    "dsv2lite-decode-T8": ("dsv2lite", 8, "decode"),
    "dsv2lite-decode-T1": ("dsv2lite", 1, "decode"),
    "granite-decode-T1": ("granite", 1, "decode"),
    "granite-prefill-T1024": ("granite", 1024, "prefill"),
    "mixtral-decode-T1": ("mixtral", 1, "decode"),
    "mixtral-decode-T8": ("mixtral", 8, "decode"),
    "mixtral-decode-T32": ("mixtral", 32, "decode"),
    "mixtral-floe10-decode-T1": ("mixtral", 1, "decode", 0.1),
    "mixtral-floe10-decode-T8": ("mixtral", 8, "decode", 0.1),
    "qwen2-prefill-T4096": ("qwen2", 4096, "prefill"),
    "dsv2lite-prefill-T4096": ("dsv2lite", 4096, "prefill"),
    "dsv2lite-cache-decode-T1": ("dsv2lite", 1, "decode"),
    "dsv2lite-lookahead-decode-T8": ("dsv2lite", 8, "decode"),
    "dsv2lite-bitslice4-draft-T1": ("dsv2lite", 1, "decode"),
    "dsv2lite-hetero-decode-T8": ("dsv2lite", 8, "decode"),
    "dsv2lite-cache-exact-decode-T1": ("dsv2lite", 1, "decode"),
}
# Multi-step decode with a persistent expert cache (ELMoE-3D heat map with
# decay): the layer runs every step with resident = the cache, which
# moe_cache_update then refreshes from the step's routed experts.
# name -> (cache capacity, heat decay, distinct one-token steps replayed)
CACHE_WORKLOADS = {"dsv2lite-cache-decode-T1": (24, 0.99, 64)}
# The same cache under the EXACT policy: every miss computed exactly, so a step
# waits for its missing experts (a stall unless their admission copy was already
# in flight).  name -> (capacity, decay, distinct one-token steps replayed)
CACHE_EXACT_WORKLOADS = {"dsv2lite-cache-exact-decode-T1": (24, 0.99, 64)}
# Decode with SPICE's confidence-aware look-ahead: every step also predicts
# the expert sets of the next J layers from the step's hidden state
# (moe_prefetch_depth over the synthetic stack's look-ahead routers).
# name -> (look-ahead layers J, confidence threshold tau, minimum depth d_min)
LOOKAHEAD_WORKLOADS = {"dsv2lite-lookahead-decode-T8": (4, 0.3, 1)}
PCIE4_X16_BYTES_PER_S = 32e9
# the cost model of the oracle's HETERO step (reference arm, CPU baseline):
# a 17.3 MB expert over PCIe 4.0 x16, 5 us on the GPU, 200 us per host row
PCIE4_HETERO_COST = dict(link_bps=PCIE4_X16_BYTES_PER_S, expert_bytes=17301504.0, gpu_expert_s=5e-6,
                         cpu_row_s=200e-6, hidden_bytes=4096.0)
# Draft layer with ELMoE-3D bit-sliced expert weights: per token, the router
# (bf16) picks the top-k experts, whose FFN (and the shared experts') runs on
# the top b bit planes of INT8 weights (moe_bitslice_ffn).  name -> b
BITSLICE_WORKLOADS = {"dsv2lite-bitslice4-draft-T1": 4}  # the host link of the pages' offloading setups
# SPICE's heterogeneous orchestration: high-confidence misses (router prob >=
# gamma) computed exactly, each missing expert fetched or run on the host cores
# by the per-miss cost model with parameters measured in the same run; also run
# with the link of the pages' PCIe 4.0 x16 setups.  name -> None
HETERO_WORKLOADS = {"dsv2lite-hetero-decode-T8": None}
DEFAULT_WORKLOAD = "dsv2lite-decode-T8"
METRIC = "MoE-layer tokens/sec (decode & prefill) and % of HBM/tensor roofline, 1xGB300"
FALLBACK_HBM_GBS = 6800.0
# nominal figures of the part, reported beside the measured-peak fractions:
# HBM3e at about 8 TB/s, dense (no 2:4 sparsity) bf16 tensor throughput
NOMINAL_HBM_GBS = 8000.0
NOMINAL_BF16_TFLOPS = 2250.0
L2_BYTES = 129 * 1024 * 1024
# The prefill half of the default line: the largest single-GPU layer shape
PREFILL_WORKLOAD = "qwen2-prefill-T4096"
CLOCK_WINDOW_S = 1.2


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=4000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(WORKLOADS))
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-prefill", action="store_true",
                   help="default workload only: skip the prefill half of the line")
    p.add_argument("--clock-window", type=float, default=CLOCK_WINDOW_S,
                   help="seconds of replays around the timed steps while clocks are sampled "
                        "(0 for profiler runs: the timed steps alone)")
    p.add_argument("--cpu-seconds", type=float, default=12.0)
    p.add_argument("--plane-copies", type=int, default=0,
                   help="bit-sliced workloads: rotating copies of the planes (0: enough to defeat L2; "
                        "small values make small cases for profiling)")
    return p.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            P = json.load(f)
        return float(P["hbm_gbs"]), float(P.get("bf16_tflops", 1900.0)), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, 1900.0, "fallback"


def sustained_bf16_tflops():
    """The measured bf16 GEMM rate back to back for seconds under the power
    cap (the denominator for work timed inside a long loop), else the
    fallback's sustained figure."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops_sustained"]), "measured bf16 sustained"
    except Exception:
        return 1700.0, "fallback bf16 sustained"


def recorded_traffic(kernel_src: str, workload: str):
    """Per-launch DRAM bytes (read + write) of the FFN stage from the committed
    ncu summary for this workload, if the kernel source and the shared header
    are unchanged since the counters were taken (else None)."""
    h = hashlib.sha256()
    srcs = (kernel_src, "common.cuh") + (("tc_common.cuh",) if kernel_src.startswith("ffn_tc") else ())
    for src in srcs:
        with open(os.path.join(ROOT, "expert_routing_ffn_gb300", "csrc", src), "rb") as f:
            h.update(f.read())
    sha = h.hexdigest()[:16]
    prof = os.path.join(ROOT, "profiles")
    if not os.path.isdir(prof):
        return None
    for name in sorted(os.listdir(prof)):
        if not name.endswith(".md"):
            continue
        with open(os.path.join(prof, name)) as f:
            txt = f.read()
        m = re.search(r"traffic_per_launch_bytes:\s*([0-9.eE+]+)\s+source_sha256_16:\s*([0-9a-f]+)"
                      r"\s+workload:\s*(\S+)", txt)
        if m and m.group(2) == sha and m.group(3) == workload:
            return float(m.group(1))
    return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 100 ms."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out = ""
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        sm, smax, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in getattr(self, "lines", []):
            f = [v.strip() for v in ln.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[0]))
                smax = max(smax, float(f[1]))
            except ValueError:
                continue
            for nm, v in zip(names, f[4:8]):
                if v.lower() in ("active", "0x1"):
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": smax or None, "reasons": sorted(reasons), "samples": len(sm)}


def timed_replays(replay, n_graphs, steps, stream, dev, world, window_s=CLOCK_WINDOW_S):
    """Time exactly `steps` replays (replay(i) replays graph i % n_graphs) with
    CUDA events on `stream`, between barriers, and sample the clocks over a
    window of at least `window_s` seconds that contains the timed steps: the
    same graphs are replayed, untimed, for about window_s before the timed
    steps and a quarter of it after them (more warm-up under the same load).
    Returns (slowest rank's ms for the timed steps, clock summary)."""
    import torch
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(n_graphs):
        replay(i)
    torch.cuda.synchronize()
    est = max(1e-6, (time.perf_counter() - t0) / n_graphs)
    pre = int(min(200_000, math.ceil(window_s / est)))
    post = int(min(50_000, math.ceil(0.25 * window_s / est)))
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(dev.index or 0) as clk:
        for i in range(pre):
            replay(i)
        torch.cuda.synchronize()
        barrier(world)
        torch.cuda.synchronize()
        ev0.record(stream)
        for i in range(steps):
            replay(i)
        ev1.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        for i in range(post):
            replay(i)
        torch.cuda.synchronize()
    ms_total = max_over_ranks(world, ev0.elapsed_time(ev1))
    summ = clk.summary()
    summ["window"] = f"{pre} untimed + {steps} timed + {post} untimed replays of the same step"
    return ms_total, summ


def fractions(achieved: float, peak: float, nominal: float, peak_src: str) -> dict:
    """Achieved against the measured peak (the roofline fraction) and against
    the part's nominal figure, each labelled."""
    return {"frac": achieved / peak, "peak": peak, "peak_source": peak_src,
            "nominal_peak": nominal, "frac_of_nominal": achieved / nominal}


def dist_setup(n_gpus):
    """Rank bookkeeping from the torchrun environment.  One process per GPU
    (NCCL); without CUDA (the multi-process tests on CPU) the gloo backend."""
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    cuda = torch.cuda.is_available()
    if world > 1:
        import torch.distributed as dist
        if cuda:
            torch.cuda.set_device(local)
        dist.init_process_group("nccl" if cuda else "gloo")
    elif cuda:
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(world, v: float) -> float:
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_batch(rank: int, i: int) -> int:
    """Token batch id of layer copy i on a rank: every replica its own tokens."""
    return 1000 * rank + i


def whole_job_tokens_per_s(world: int, T: int, steps: int, ms_max: float) -> float:
    """Tokens all ranks processed / the slowest rank's time (weak scaling)."""
    return world * T * steps / (ms_max / 1e3)


def oracle_step(cfg, W, x, wl_name):
    """One step of the workload through the float64 oracle: the layer forward,
    and for a look-ahead workload the prefetch depth over its look-ahead
    routers."""
    import oracle
    if wl_name in HETERO_WORKLOADS:
        oracle.layer_forward(cfg, W, x, policy=oracle.POL_HETERO, cost=PCIE4_HETERO_COST)
        return
    if wl_name in CACHE_EXACT_WORKLOADS:
        oracle.layer_forward(cfg, W, x, policy=0)
        return
    oracle.layer_forward(cfg, W, x)
    la = LOOKAHEAD_WORKLOADS.get(wl_name)
    if la:
        Ws, bs = make_lookahead_routers(cfg, la[0])
        oracle.prefetch_depth(x, Ws, bs, cfg.k, la[1], la[2])


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def cpu_baseline(cfg, W, T, seconds, batch_offset=0, wl_name=None):
    """The float64 oracle, as it stands, on a bounded sample of the workload,
    on every core of the process's affinity mask, plus a single-thread figure.

    Decode (T <= 64): whole T-token batches, as many running at once as the
    cores allow (one OpenMP thread per token), until `seconds` have passed.
    Prefill: tokens of one T-token batch (its batch resident set computed once,
    beforehand), in chunks of one token per core, until `seconds` have passed."""
    import oracle
    from concurrent.futures import ThreadPoolExecutor
    cores = host_cores()
    base_threads = oracle.num_threads()

    def run_decode(threads, budget, offset):
        par = max(1, threads // T)

        def one(b):
            oracle.set_num_threads(min(T, threads))
            oracle_step(cfg, W, make_tokens(cfg, T=T, batch=10_000 + batch_offset + offset + b), wl_name)
            return T

        n_tok, b, t0 = 0, 0, time.perf_counter()
        with ThreadPoolExecutor(par) as ex:
            while True:
                n_tok += sum(ex.map(one, range(b, b + par)))
                b += par
                el = time.perf_counter() - t0
                if el >= budget:
                    break
        return n_tok, el, b, min(T, threads) * par

    def run_prefill(threads, budget, x, resident, order):
        oracle.set_num_threads(threads)
        n_tok, t0 = 0, time.perf_counter()
        while n_tok < len(order):
            rows = np.sort(order[n_tok:n_tok + threads])
            oracle.layer_forward(cfg, W, x[rows], resident=resident)
            n_tok += len(rows)
            el = time.perf_counter() - t0
            if el >= budget:
                break
        return n_tok, el

    try:
        if T <= 64:
            n, el, b, used = run_decode(cores, seconds, 0)
            n1, el1, b1, _ = run_decode(1, max(1.0, seconds / 4), 50_000)
            res = {"value": n / el, "unit": "tokens/s", "cores": used, "kind": "oracle",
                   "sample": f"{b} batches of {T} tokens ({n} tokens, {el:.1f} s) through the float64 CPU "
                             f"oracle, {max(1, cores // T)} batches at a time, OpenMP over the tokens of a "
                             f"batch; {cores} cores in the affinity mask",
                   "single_thread": {"value": n1 / el1, "unit": "tokens/s", "cores": 1,
                                     "sample": f"{b1} batches of {T} tokens ({n1} tokens, {el1:.1f} s), "
                                               f"one thread"}}
        else:
            x = make_tokens(cfg, T=T, batch=10_000 + batch_offset)
            resident, _ = oracle.resident_mask(cfg, W, x)
            order = np.random.default_rng(batch_offset).permutation(T)
            n, el = run_prefill(cores, seconds, x, resident, order)
            n1, el1 = run_prefill(1, max(2.0, seconds / 4), x, resident, order[::-1].copy())
            res = {"value": n / el, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                   "sample": f"{n} of the {T} tokens of one prefill batch (seeded sample, {el:.1f} s) through "
                             f"the float64 CPU oracle, {cores} tokens at a time (OpenMP over tokens), the "
                             f"batch resident set computed beforehand; {cores} cores in the affinity mask",
                   "single_thread": {"value": n1 / el1, "unit": "tokens/s", "cores": 1,
                                     "sample": f"{n1} tokens of the same batch ({el1:.1f} s), one thread"}}
    finally:
        oracle.set_num_threads(base_threads)
    return res


class BitsliceOracle:
    """The draft layer of a bit-sliced workload through the float64 oracle:
    router softmax and top-k, then the gate-weighted b-bit expert FFNs of the
    routed experts plus the shared experts."""

    def __init__(self, cfg, W, bits):
        import oracle
        self.o, self.cfg, self.W, self.bits, self.q = oracle, cfg, W, bits, {}

    def _q(self, key, Wg, Wu, Wd):
        if key not in self.q:
            o = self.o
            self.q[key] = (o.bitslice_quantize(Wg) + o.bitslice_quantize(Wu) + o.bitslice_quantize(Wd, transpose=True))
        return self.q[key]

    def token(self, x):
        o, cfg, W = self.o, self.cfg, self.W
        lg = o.logits(x[None], W.w_router, W.router_bias)[0]
        p = o.softmax(lg[None])[0]
        y = np.zeros(cfg.d)
        for e in o.topk(lg, cfg.k):
            e = int(e)
            y += p[e] * o.bitslice_ffn(x, *self._q(("r", e), W.w_gate[e], W.w_up[e], W.w_down[e]), self.bits)
        for sh in range(cfg.n_shared):
            y += o.bitslice_ffn(x, *self._q(("s", sh), W.sh_gate[sh], W.sh_up[sh], W.sh_down[sh]), self.bits)
        return y


def workload_cfg(wl_name):
    """(layer config, tokens per step, phase) of a named workload."""
    cfg_name, T, phase = WORKLOADS[wl_name][:3]
    cfg = CONFIGS[cfg_name]
    if len(WORKLOADS[wl_name]) > 3:
        cfg = cfg.with_(keep_frac=WORKLOADS[wl_name][3])
    return cfg, T, phase


def reference_line(args, wl_name, steps, warmup, budget=120.0):
    """Reference arm: the float64 oracle timed on the host cores, one bounded
    sample of the workload per step (at most 32 tokens of the batch, every
    core of the affinity mask), for at most `budget` seconds."""
    import oracle
    cfg, T, phase = workload_cfg(wl_name)
    if wl_name in BITSLICE_WORKLOADS:
        W = make_weights(cfg)
        bo = BitsliceOracle(cfg, W, BITSLICE_WORKLOADS[wl_name])
        warm = min(warmup, 3)
        for i in range(warm):
            bo.token(make_tokens(cfg, T=1, batch=20_000 + i)[0])
        t0, n = time.perf_counter(), 0
        while n < steps:
            bo.token(make_tokens(cfg, T=1, batch=30_000 + n)[0])
            n += 1
            if time.perf_counter() - t0 > budget:
                break
        el = time.perf_counter() - t0
        value = n / el
        return {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": 1, "steps": n,
                "warmup": warm, "ms_per_step": 1e3 * el / n, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "impl": "reference", "config": {"workload": wl_name, "tokens_per_step": 1},
                "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                                 "sample": f"{n} one-token draft steps (of {steps} requested; capped "
                                           f"at {budget:.0f} s), quantisation of the experts included"},
                "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    W = make_weights(cfg)
    cores = host_cores()
    Ts = min(T, 32)  # a step is a bounded sample of the batch (tokens are independent)
    resident = None
    if T > 64:
        # prefill: tokens of one full batch, with the batch resident set of that batch
        x_full = make_tokens(cfg, T=T, batch=30_000)
        resident, _ = oracle.resident_mask(cfg, W, x_full)
        order = np.random.default_rng(0).permutation(T)
        Ts = min(32, max(cores, 8))
    warm = min(warmup, 3)  # the oracle has no caches to warm beyond a first call

    def one(i):
        if resident is None:
            oracle_step(cfg, W, make_tokens(cfg, T=Ts, batch=30_000 + i), wl_name)
        else:
            rows = np.sort(order[(i * Ts) % T:(i * Ts) % T + Ts])
            oracle.layer_forward(cfg, W, x_full[rows], resident=resident)
        return Ts

    for i in range(warm):
        one(10_000 + i if resident is None else i)
    t0, n, k = time.perf_counter(), 0, 0
    while k < steps:
        n += one(k)
        k += 1
        if time.perf_counter() - t0 > budget:
            break
    el = time.perf_counter() - t0
    value = n / el
    used = min(oracle.num_threads(), Ts)
    what = (f"{k} steps of {Ts} tokens (of {steps} requested; capped at {budget:.0f} s)" if resident is None else
            f"{k} steps of {Ts} of the {T} tokens of one prefill batch (of {steps} requested; capped at "
            f"{budget:.0f} s), the batch resident set computed beforehand")
    return {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": 1, "steps": k,
            "warmup": warm, "ms_per_step": 1e3 * el / k, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "impl": "reference",
            "config": {"workload": wl_name, "tokens_per_step": Ts},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": used, "kind": "oracle",
                             "sample": what},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def run_reference(args, wl_name, rank, with_prefill=False):
    """The reference arm's line, printed by rank 0 only (the other ranks of a
    torchrun launch exit without work); with_prefill adds the prefill
    workload's oracle timing under "prefill"."""
    if rank != 0:
        return
    line = reference_line(args, wl_name, args.steps, args.warmup)
    if with_prefill:
        line["prefill"] = nested(reference_line(args, PREFILL_WORKLOAD, max(3, min(args.steps, 100)),
                                                args.warmup, budget=45.0))
    print(json.dumps(line), flush=True)


NESTED_DROP = ("metric", "n_gpus", "higher_is_better", "scaling", "vs_baseline", "data", "impl")


def nested(line: dict) -> dict:
    """A workload's line as the value of a key of another line."""
    return {k: v for k, v in line.items() if k not in NESTED_DROP}


def run_bitslice(args, wl_name, cfg, T, W, dev, world, rank, hbm_gbs, peak_src, steps, warmup):
    """Timed draft layer with b-bit bit-sliced expert weights (see
    BITSLICE_WORKLOADS): one step = the bf16 router (moe_route, top-k gates)
    and one moe_bitslice_ffn call over the routed and the shared experts,
    over several packed copies of the planes so that the planes one step
    reads come from HBM."""
    import torch
    import expert_routing_ffn_gb300 as moe
    bits = BITSLICE_WORKLOADS[wl_name]
    d, I, N, k, ns, Is = cfg.d, cfg.I, cfg.N, cfg.k, cfg.n_shared, cfg.I_shared
    assert Is == I or ns == 0
    dt = torch.bfloat16
    step_bytes = (k + ns) * 3 * I * d * bits / 8
    n_copies = int(min(8, max(2, math.ceil(1 + 2 * L2_BYTES / step_bytes))))
    if args.plane_copies > 0:
        n_copies = args.plane_copies
    w8 = 8 * I * d // 32

    def pack_set(mats, n):
        P = [torch.zeros(n * w8, dtype=torch.int32, device=dev) for _ in range(3)]
        S = [torch.zeros(n * (I if m < 2 else d), dtype=torch.float32, device=dev) for m in range(3)]
        for e in range(n):
            for m in range(3):
                w = torch.from_numpy(mats[m][e]).to(dev).to(dt)
                R = I if m < 2 else d
                moe.moe_bitslice_pack(w, m == 2, P[m][e * w8:(e + 1) * w8], S[m][e * R:(e + 1) * R])
        return P, S

    # the routed experts, then the shared experts, back to back
    cat = lambda a, b: np.concatenate([a, b]) if ns else a
    planes = pack_set((cat(W.w_gate, W.sh_gate), cat(W.w_up, W.sh_up), cat(W.w_down, W.sh_down)), N + ns)
    torch.cuda.synchronize()
    # further copies of every plane at distinct addresses (the same values)
    copies = [planes] + [([t.clone() for t in planes[0]], planes[1]) for _ in range(n_copies - 1)]
    dims = moe.make_dims(T, d, N, k, I, ns, Is, cfg.r, wtype=cfg.wtype)
    ws = torch.zeros(moe.moe_workspace_size(dims), dtype=torch.uint8, device=dev)
    w_router = torch.from_numpy(W.w_router).to(dev).to(dt)
    bias = None if W.router_bias is None else torch.from_numpy(W.router_bias).to(dev)
    n_x = 64
    xs = [torch.from_numpy(make_tokens(cfg, T=T, batch=replica_batch(rank, i))).to(dev).to(dt).contiguous()
          for i in range(n_x)]
    topk_idx = torch.zeros((T, k), dtype=torch.int32, device=dev)
    topk_gate = torch.zeros((T, k), dtype=torch.float32, device=dev)
    prob = torch.zeros((T, N), dtype=torch.float32, device=dev)
    dhat = torch.zeros(T, dtype=torch.int32, device=dev)
    pmask = torch.zeros(T, dtype=torch.int64, device=dev)
    y = torch.zeros((T, d), dtype=torch.float32, device=dev)
    scratch = torch.zeros(moe.moe_bitslice_scratch_size(d, I, T, k + ns), dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(device=dev)
    torch.cuda.set_stream(stream)

    def ffn(c):
        P, S = copies[c % n_copies]
        moe.moe_bitslice_ffn(d, I, N, bits, xs_cur[0], topk_idx, topk_gate, P[0], S[0], P[1], S[1], P[2], S[2], y,
                             scratch, n_shared=ns, stream=stream)

    xs_cur = [xs[0]]

    def step(i):
        xs_cur[0] = xs[i % n_x]
        moe.moe_route(dims, xs_cur[0], w_router, bias, None, None, None, None, cfg.tau, 0, topk_idx, topk_gate,
                      prob, dhat, pmask, None, None, ws, stream)
        ffn(i)

    for i in range(max(warmup, n_copies)):
        step(i)
    st, det = moe.moe_check(ws)
    if st != moe.MOE_OK:
        raise RuntimeError(f"device error {moe.status_string(st)} ({det})")
    n_graphs = max(n_copies, n_x)
    graphs = []
    n0 = moe.moe_launch_total()
    for c in range(n_graphs):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            step(c)
        graphs.append(g)
    launches_per_step = (moe.moe_launch_total() - n0) // n_graphs
    for i in range(warmup):
        graphs[i % n_graphs].replay()
    torch.cuda.synchronize()
    ms_total, clocks = timed_replays(lambda i: graphs[i % n_graphs].replay(), n_graphs, steps, stream, dev, world,
                                     args.clock_window)
    ms_per_step = ms_total / steps
    value = whole_job_tokens_per_s(world, T, steps, ms_total)

    # the bit-sliced FFN call alone (routing of each token batch in place):
    # algorithmic bytes = the top-b planes of the distinct routed experts and
    # the shared experts, plus their scales
    n_k = max(50, min(2000, steps // 2))
    fb = []
    for c in range(n_x):
        step(c)
        torch.cuda.synchronize()
        u = len(set(topk_idx.cpu().numpy().ravel().tolist()))
        fb.append((u + ns) * (3 * I * d * bits / 8 + 4 * (2 * I + d)))
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_k)]
    for i in range(n_k):
        c = i % n_x
        xs_cur[0] = xs[c]
        moe.moe_route(dims, xs[c], w_router, bias, None, None, None, None, cfg.tau, 0, topk_idx, topk_gate,
                      prob, dhat, pmask, None, None, ws, stream)
        evs[i][0].record(stream)
        ffn(i)
        evs[i][1].record(stream)
    torch.cuda.synchronize()
    k_ms = [a.elapsed_time(b) for a, b in evs]
    k_bytes = [fb[i % n_x] for i in range(n_k)]
    med_ms = statistics.median(k_ms)
    achieved = statistics.mean(k_bytes) / (med_ms / 1e3) / 1e9
    roof = {"kernel": "moe_bitslice_ffn (bitslice_gateup_kernel + bitslice_down_kernel with the gated slot sum)",
            "ffn_path": f"bitslice-b{bits}", "bound": "hbm", "achieved": achieved, "unit": "GB/s",
            **fractions(achieved, hbm_gbs, NOMINAL_HBM_GBS, peak_src),
            "algorithmic_bytes_per_launch": float(statistics.mean(fb)), "median_launch_ms": med_ms,
            "avg_launch_ms": statistics.mean(k_ms), "launches_timed": n_k, "traffic": None}

    # end to end: pinned host x -> device, draft layer, y -> pinned host, every step
    x_host = [xs[c].cpu().pin_memory() for c in range(n_x)]
    y_host = torch.empty_like(y, device="cpu").pin_memory()
    n_e2e = max(20, min(steps, 1000))
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(n_e2e):
        xs[i % n_x].copy_(x_host[i % n_x], non_blocking=True)
        step(i)
        y_host.copy_(y, non_blocking=True)
        stream.synchronize()
    e2e_s = max_over_ranks(world, time.perf_counter() - t0)
    e2e_value = world * T * n_e2e / e2e_s
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": steps,
        "warmup": warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": f"b{bits} bit planes of int8 (f32 accumulate)",
        "data": "synthetic (seeded N(0,0.02^2) weights, N(0,1) tokens; shapes of the named model)",
        "config": {"workload": wl_name, "tokens_per_step": T, "d": d, "experts": N, "top_k": k,
                   "intermediate": I, "shared_experts": ns, "bits": bits, "parallelism": f"replicas x{world}",
                   "l2": f"inputs larger than L2: {n_copies} rotating copies of every expert's planes",
                   "cuda_graph": True},
        "roofline": roof,
        "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": xs[0].numel() * xs[0].element_size(),
                "d2h_bytes_per_step": y.numel() * 4, "steps": n_e2e,
                "note": "moe_route + moe_bitslice_ffn per step with pinned-host copies and a stream sync, no graph"},
        "gpu_launches": int(launches_per_step * steps),
        "clocks": clocks,
    }
    if rank == 0 and not args.no_cpu_baseline:
        bo = BitsliceOracle(cfg, W, bits)
        bo.token(make_tokens(cfg, T=1, batch=10_000)[0])  # quantises the experts it reads
        n_tok, t0 = 0, time.perf_counter()
        while True:
            bo.token(make_tokens(cfg, T=1, batch=10_001 + n_tok)[0])
            n_tok += 1
            el = time.perf_counter() - t0
            if el >= args.cpu_seconds:
                break
        line["cpu_baseline"] = {"value": n_tok / el, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                                "sample": f"{n_tok} one-token draft steps ({el:.1f} s) through the float64 "
                                          f"oracle, single thread, experts quantised beforehand when first read"}
    return line


def run_hetero(args, wl_name, cfg, T, W, dev, world, rank, hbm_gbs, peak_src, steps, warmup):
    """Timed layer steps on the heterogeneous CPU-GPU path
    (moe_layer_forward_hetero): the cost model's parameters are measured
    first (the host link by expert copies, the GPU time of one expert from
    the decode FFN stage, the host time of one expert row from
    moe_cpu_experts), then the layer runs with them and again with the link
    of a PCIe 4.0 x16 setup.  A step is host-orchestrated (the host waits for
    the decisions), so it is timed on the host clock around synchronised
    steps; the LoRE/substitute-only policy (HYBRID) is timed the same way
    for comparison."""
    import torch
    import expert_routing_ffn_gb300 as moe
    from expert_routing_ffn_gb300.layer import DeviceLayer, HeteroHost, LayerBuffers, forward, forward_hetero
    esize = 2
    expert_bytes = 3 * cfg.I * cfg.d * esize
    layer = DeviceLayer(cfg, W, T, device=str(dev))
    host = HeteroHost(layer, T)
    bufs = LayerBuffers(layer, T)
    stream = torch.cuda.Stream(device=dev)
    torch.cuda.set_stream(stream)
    side = torch.cuda.Stream(device=dev)
    ev = torch.cuda.Event()
    n_x = 64
    xs = [torch.from_numpy(make_tokens(cfg, T=T, batch=replica_batch(rank, i))).to(dev).to(layer.dt).contiguous()
          for i in range(n_x)]
    D = layer.dims.with_T(T)

    # link: 8 experts from pinned host memory
    mask = (1 << 8) - 1
    moe.moe_stage_experts(D, mask, host.w_gate, host.w_up, host.w_down, list(layer.w_gate), list(layer.w_up),
                          list(layer.w_down), side, ev)
    side.synchronize()
    t0 = time.perf_counter()
    for _ in range(3):
        nb = moe.moe_stage_experts(D, mask, host.w_gate, host.w_up, host.w_down, list(layer.w_gate),
                                   list(layer.w_up), list(layer.w_down), side, ev)
    side.synchronize()
    link = 3 * nb / (time.perf_counter() - t0)
    # GPU time of one expert: the decode FFN stage's bytes per second applied to one expert
    forward(layer, bufs, xs[0], stream=stream)
    torch.cuda.synchronize()
    off = bufs.expert_offsets.cpu().numpy()
    u = int((np.diff(off) > 0).sum())
    ffn_bytes = u * expert_bytes + cfg.n_shared * 3 * cfg.I_shared * cfg.d * esize
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(30)]
    for a, b in evs:
        a.record(stream)
        moe.moe_expert_ffn(D, xs[0], layer.table, bufs.expert_offsets, bufs.perm, 1.0, bufs.y_perm, bufs.y_shared,
                           layer.ws, stream)
        b.record(stream)
    torch.cuda.synchronize()
    ffn_ms = statistics.median([a.elapsed_time(b) for a, b in evs])
    gpu_expert_s = expert_bytes / (ffn_bytes / (ffn_ms / 1e3))
    # host time of one expert row: moe_cpu_experts on one host slot
    hk = torch.zeros((T, cfg.k), dtype=torch.int32)
    hi = torch.zeros((T, cfg.k), dtype=torch.int32)
    for t in range(T):
        hi[t] = torch.arange(cfg.k, dtype=torch.int32) + t
    hk[0, 0] = moe.MOE_KIND_CPU
    host.x.copy_(xs[0].cpu())
    times = []
    for _ in range(12):
        t1 = time.perf_counter()
        moe.moe_cpu_experts(D, host.x, hi, hk, host.w_gate, host.w_up, host.w_down, host.y_rows, host.scratch)
        times.append(time.perf_counter() - t1)
    cpu_row_s = statistics.median(times[2:])
    measured = dict(link_bps=link, expert_bytes=float(expert_bytes), gpu_expert_s=gpu_expert_s,
                    cpu_row_s=cpu_row_s, hidden_bytes=float(cfg.d * esize))
    pcie = dict(measured, link_bps=PCIE4_X16_BYTES_PER_S)

    def lib_cost(c):
        return moe.hetero_cost(c["link_bps"], c["expert_bytes"], c["gpu_expert_s"], c["cpu_row_s"], c["hidden_bytes"])

    def timed(cost, n):
        cst = lib_cost(cost)
        acc = {"cpu_slots": 0, "fetch_experts": 0, "lore_slots": 0, "fetch_bytes": 0.0, "cpu_link_bytes": 0.0,
               "host_ms": 0.0, "wait_ms": 0.0}
        for i in range(max(3, warmup)):
            forward_hetero(layer, bufs, xs[i % n_x], host, cst, side, ev, stream=stream)
        stream.synchronize()
        t1 = time.perf_counter()
        for i in range(n):
            st = forward_hetero(layer, bufs, xs[i % n_x], host, cst, side, ev, stream=stream)
            stream.synchronize()
            for key in acc:
                acc[key] += getattr(st, key)
        el = time.perf_counter() - t1
        res = {"tokens_per_s": T * n / el, "ms_per_step": 1e3 * el / n, "steps": n,
               "fetch_min_rows": moe.moe_hetero_fetch_min_rows(cst)}
        res.update({f"{key}_per_step": v / n for key, v in acc.items()})
        return res, el

    n_steps = max(20, min(steps, 400))
    barrier(world)
    with ClockSampler(dev.index or 0) as clk:
        main_res, el = timed(measured, n_steps)
    clocks = clk.summary()
    barrier(world)
    pcie_res, _ = timed(pcie, n_steps)
    # the LoRE/substitute-only policy, eager and synchronised the same way
    for i in range(3):
        forward(layer, bufs, xs[i % n_x], stream=stream)
    stream.synchronize()
    t1 = time.perf_counter()
    for i in range(n_steps):
        forward(layer, bufs, xs[i % n_x], stream=stream)
        stream.synchronize()
    hybrid_tps = T * n_steps / (time.perf_counter() - t1)
    st, det = moe.moe_check(layer.ws)
    if st != moe.MOE_OK:
        raise RuntimeError(f"device error {moe.status_string(st)} ({det})")

    # end to end: pinned host x -> device, the hetero step, out -> pinned host
    x_host = [xs[c].cpu().pin_memory() for c in range(n_x)]
    out_host = torch.empty_like(bufs.out, device="cpu").pin_memory()
    cst = lib_cost(measured)
    t1 = time.perf_counter()
    for i in range(n_steps):
        xs[i % n_x].copy_(x_host[i % n_x], non_blocking=True)
        forward_hetero(layer, bufs, xs[i % n_x], host, cst, side, ev, stream=stream)
        out_host.copy_(bufs.out, non_blocking=True)
        stream.synchronize()
    e2e_value = world * T * n_steps / max_over_ranks(world, time.perf_counter() - t1)
    value = world * T * n_steps / max_over_ranks(world, el)
    ach = ffn_bytes / (ffn_ms / 1e3) / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": n_steps,
        "warmup": max(3, warmup), "ms_per_step": main_res["ms_per_step"], "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,0.02^2) weights, N(0,1) tokens; shapes of the named model)",
        "config": {"workload": wl_name, "tokens_per_step": T, "d": cfg.d, "experts": cfg.N, "top_k": cfg.k,
                   "intermediate": cfg.I, "shared_experts": cfg.n_shared, "miss_policy": "hetero",
                   "gamma": cfg.gamma, "resident": cfg.n_resident, "parallelism": f"replicas x{world}",
                   "timing": "host clock around synchronised steps (the host waits for each step's decisions)",
                   "l2": "one layer copy; every fetched expert is copied in from pinned host memory each step"},
        "roofline": {"kernel": "moe_expert_ffn (decode FFN stage of this layer, timed alone)", "bound": "hbm",
                     "achieved": ach, "unit": "GB/s", **fractions(ach, hbm_gbs, NOMINAL_HBM_GBS, peak_src),
                     "algorithmic_bytes_per_launch": float(ffn_bytes), "median_launch_ms": ffn_ms,
                     "traffic": None},
        "hetero": {"cost_measured": measured, "measured_link": main_res, "pcie4_x16_link": dict(pcie_res, cost=pcie),
                   "hybrid_policy_tokens_per_s": hybrid_tps,
                   "note": "cpu slots, fetched experts and link bytes per step; HYBRID = LoRE or substitute for "
                           "every miss (no exact miss), the same host-synchronised loop"},
        "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": xs[0].numel() * 2,
                "d2h_bytes_per_step": bufs.out.numel() * 4, "steps": n_steps,
                "note": "moe_layer_forward_hetero per step with pinned-host copies of x and out"},
        "clocks": clocks,
        "gpu_launches": None,
    }
    n0 = moe.moe_launch_total()
    forward_hetero(layer, bufs, xs[0], host, cst, side, ev, stream=stream)
    stream.synchronize()
    line["gpu_launches"] = int((moe.moe_launch_total() - n0) * n_steps)
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(cfg, W, T, args.cpu_seconds, wl_name=wl_name)
    return line


def run_cache_exact(args, wl_name, cfg, T, W, dev, world, rank, hbm_gbs, peak_src, steps, warmup):
    """Decode steps over the overlapped expert cache under the EXACT policy
    (moe_cache_step): misses are computed exactly, so a step whose missing
    experts were not already admitted and in flight waits for their copies.
    Host clock around the steps (the host reads each step's fetch mask)."""
    import torch
    import expert_routing_ffn_gb300 as moe
    from expert_routing_ffn_gb300.layer import CachePipeline, DeviceLayer, LayerBuffers, forward
    capacity, decay, n_x = CACHE_EXACT_WORKLOADS[wl_name]
    expert_bytes = 3 * cfg.I * cfg.d * 2
    layer = DeviceLayer(cfg, W, T, device=str(dev))
    bufs = LayerBuffers(layer, T)
    stream = torch.cuda.Stream(device=dev)
    torch.cuda.set_stream(stream)
    xs = [torch.from_numpy(make_tokens(cfg, T=T, batch=replica_batch(rank, i))).to(dev).to(layer.dt).contiguous()
          for i in range(n_x)]
    pipe = CachePipeline(layer, capacity, decay, stream=stream)
    pipe.start((1 << capacity) - 1)
    for i in range(max(3, warmup)):
        pipe.step(bufs, xs[i % n_x], policy=moe.MOE_MISS_EXACT, n_resident=0)
    stream.synchronize()
    n = max(50, min(steps, 1000))
    p = pipe.pipe
    base = (p.staged_experts, p.staged_bytes, p.in_time_experts, p.stall_experts, p.stall_steps)
    hits = slots = 0
    barrier(world)
    with ClockSampler(dev.index or 0) as clk:
        t0 = time.perf_counter()
        for i in range(n):
            pipe.step(bufs, xs[i % n_x], policy=moe.MOE_MISS_EXACT, n_resident=0)
        stream.synchronize()
        el = time.perf_counter() - t0
    clocks = clk.summary()
    barrier(world)
    d = [a - b for a, b in zip((p.staged_experts, p.staged_bytes, p.in_time_experts, p.stall_experts,
                                p.stall_steps), base)]
    st = pipe.stats.cpu().numpy()  # hits / slots since start (includes warm-up)
    hits, slots = int(st[0]), int(st[1])
    # end to end with pinned-host copies of x and out every step
    x_host = [xs[c].cpu().pin_memory() for c in range(n_x)]
    out_host = torch.empty_like(bufs.out, device="cpu").pin_memory()
    t1 = time.perf_counter()
    for i in range(n):
        xs[i % n_x].copy_(x_host[i % n_x], non_blocking=True)
        pipe.step(bufs, xs[i % n_x], policy=moe.MOE_MISS_EXACT, n_resident=0)
        out_host.copy_(bufs.out, non_blocking=True)
        stream.synchronize()
    e2e_s = time.perf_counter() - t1
    pipe.drain()
    stt, det = moe.moe_check(layer.ws)
    if stt != moe.MOE_OK:
        raise RuntimeError(f"device error {moe.status_string(stt)} ({det})")
    # the FFN stage of this layer, timed alone (all experts on the device)
    forward(layer, bufs, xs[0], stream=stream, policy=moe.MOE_MISS_EXACT)
    torch.cuda.synchronize()
    off = bufs.expert_offsets.cpu().numpy()
    ffn_bytes = int((np.diff(off) > 0).sum()) * expert_bytes + cfg.n_shared * 3 * cfg.I_shared * cfg.d * 2
    D = layer.dims.with_T(T)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(50)]
    for a, b in evs:
        a.record(stream)
        moe.moe_expert_ffn(D, xs[0], layer.table, bufs.expert_offsets, bufs.perm, 1.0, bufs.y_perm, bufs.y_shared,
                           layer.ws, stream)
        b.record(stream)
    torch.cuda.synchronize()
    ffn_ms = statistics.median([a.elapsed_time(b) for a, b in evs])
    ach = ffn_bytes / (ffn_ms / 1e3) / 1e9
    step_s = el / n
    link = d[1] / max(1e-9, el) if d[1] else None
    line = {
        "metric": METRIC, "value": world * T * n / max_over_ranks(world, el), "unit": "tokens/s", "n_gpus": world,
        "steps": n, "warmup": max(3, warmup), "ms_per_step": 1e3 * step_s, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,0.02^2) weights, N(0,1) tokens; shapes of the named model)",
        "config": {"workload": wl_name, "tokens_per_step": T, "d": cfg.d, "experts": cfg.N, "top_k": cfg.k,
                   "intermediate": cfg.I, "shared_experts": cfg.n_shared, "miss_policy": "exact",
                   "resident": f"expert cache of {capacity} (heat decay {decay})",
                   "parallelism": f"replicas x{world}",
                   "timing": "host clock around the steps (each EXACT step reads its fetch mask on the host)"},
        "roofline": {"kernel": "moe_expert_ffn (decode FFN stage of this layer, timed alone)", "bound": "hbm",
                     "achieved": ach, "unit": "GB/s", **fractions(ach, hbm_gbs, NOMINAL_HBM_GBS, peak_src),
                     "algorithmic_bytes_per_launch": float(ffn_bytes), "median_launch_ms": ffn_ms, "traffic": None},
        "cache": {"capacity": capacity, "decay": decay, "hit_rate": hits / max(1, slots),
                  "stall_rate": d[4] / n, "stalled_experts_per_step": d[3] / n,
                  "in_time_experts_per_step": d[2] / n, "copied_experts_per_step": d[0] / n,
                  "copied_bytes_per_step": d[1] / n,
                  "d_min_measured_link": (moe.moe_prefetch_min_depth(expert_bytes, link, step_s) if link else None),
                  "d_min_pcie4_x16": moe.moe_prefetch_min_depth(expert_bytes, PCIE4_X16_BYTES_PER_S, step_s),
                  "note": "stall = a step that copied a missing expert on demand and waited for it; in time = a "
                          "miss whose admission copy was already in flight or landed (the GPU waits only on its "
                          "event); hit rate over all steps since the start"},
        "e2e": {"value": world * T * n / max_over_ranks(world, e2e_s), "unit": "tokens/s",
                "h2d_bytes_per_step": xs[0].numel() * 2 + d[1] / n, "d2h_bytes_per_step": bufs.out.numel() * 4 + 40,
                "steps": n, "note": "moe_cache_step per step with pinned-host copies of x and out"},
        "clocks": clocks,
        "gpu_launches": None,
    }
    n0 = moe.moe_launch_total()
    pipe.step(bufs, xs[0], policy=moe.MOE_MISS_EXACT, n_resident=0)
    stream.synchronize()
    line["gpu_launches"] = int((moe.moe_launch_total() - n0) * n)
    pipe.drain()
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(cfg, W, T, args.cpu_seconds, wl_name=wl_name)
    return line


def run_workload(args, wl_name, world, rank, dev, steps, warmup, with_cpu=True):
    """Measure one workload; returns its JSON line (a dict)."""
    import torch
    import expert_routing_ffn_gb300 as moe
    from expert_routing_ffn_gb300.layer import DeviceLayer, LayerBuffers, forward, forward_host

    cfg, T, phase = workload_cfg(wl_name)
    hbm_gbs, bf16_tflops, peak_src = peaks()
    W = make_weights(cfg)
    if wl_name in BITSLICE_WORKLOADS:
        return run_bitslice(args, wl_name, cfg, T, W, dev, world, rank, hbm_gbs, peak_src, steps, warmup)
    if wl_name in HETERO_WORKLOADS:
        return run_hetero(args, wl_name, cfg, T, W, dev, world, rank, hbm_gbs, peak_src, steps, warmup)
    if wl_name in CACHE_EXACT_WORKLOADS:
        return run_cache_exact(args, wl_name, cfg, T, W, dev, world, rank, hbm_gbs, peak_src, steps, warmup)
    base = DeviceLayer(cfg, W, T, device=str(dev))
    esize = 2 if cfg.wtype == "bf16" else 4
    expert_bytes = 3 * cfg.I * cfg.d * esize
    shared_bytes = cfg.n_shared * 3 * cfg.I_shared * cfg.d * esize
    layer_bytes = cfg.N * expert_bytes + shared_bytes
    # enough copies that the expert bytes of one step are pushed out of L2 (by
    # at least twice its size) before the same copy is read again
    step_bytes = min(cfg.N, T * cfg.k) * expert_bytes + shared_bytes
    n_copies = int(min(16, max(2, math.ceil(1 + 2 * L2_BYTES / step_bytes))))
    layers = [base] + [base.clone() for _ in range(n_copies - 1)]
    stream = torch.cuda.Stream(device=dev)
    torch.cuda.set_stream(stream)
    bufs = [LayerBuffers(L, T) for L in layers]
    cache_cfg = CACHE_WORKLOADS.get(wl_name)
    n_x = cache_cfg[2] if cache_cfg else n_copies  # distinct token batches replayed
    xs = [torch.from_numpy(make_tokens(cfg, T=T, batch=replica_batch(rank, i))).to(dev).to(base.dt).contiguous()
          for i in range(n_x)]
    if cache_cfg:
        # one cache for the layer: every weight copy reads the same resident mask
        capacity, decay = cache_cfg[0], cache_cfg[1]
        cache_t = torch.full((1,), (1 << capacity) - 1, dtype=torch.int64, device=dev)  # predefined start set
        heat_t = torch.zeros(cfg.N, dtype=torch.float32, device=dev)
        admit_t = torch.zeros(1, dtype=torch.int64, device=dev)
        cstats_t = torch.zeros(4, dtype=torch.int32, device=dev)
        for L in layers:
            L.resident = cache_t

    la_cfg = LOOKAHEAD_WORKLOADS.get(wl_name)
    if la_cfg:
        la_J, la_tau, la_dmin = la_cfg
        la_W, la_b = make_lookahead_routers(cfg, la_J)
        la_Wd = [torch.from_numpy(w).to(dev).to(base.dt).contiguous() for w in la_W]
        la_bd = None if la_b is None else [torch.from_numpy(b).to(dev) for b in la_b]
        la_logits = torch.zeros((la_J, T, cfg.N), dtype=torch.float32, device=dev)
        la_conf = torch.zeros((T, la_J), dtype=torch.float32, device=dev)
        la_depth = torch.zeros(T, dtype=torch.int32, device=dev)
        la_tok = torch.zeros((T, la_J), dtype=torch.int64, device=dev)
        la_lay = torch.zeros(la_J, dtype=torch.int64, device=dev)

        def lookahead(c, x):
            moe.moe_prefetch_depth(layers[c].dims.with_T(T), x, la_Wd, la_bd, la_tau, la_dmin, la_logits, la_conf,
                                   la_depth, la_tok, la_lay, layers[c].ws, stream)

    def step(i):
        c = i % n_copies
        if la_cfg:
            forward(layers[c], bufs[c], xs[c], stream=stream)
            lookahead(c, xs[c])
        elif cache_cfg:
            forward(layers[c], bufs[c], xs[i % n_x], stream=stream, n_resident=0)
            moe.moe_cache_update(layers[c].dims.with_T(T), bufs[c].topk_idx, decay, capacity, heat_t, cache_t,
                                 admit_t, cstats_t, stream)
        else:
            forward(layers[c], bufs[c], xs[c], stream=stream)

    # eager warm-up, error check, then one CUDA graph per layer copy
    for i in range(max(warmup, n_copies)):
        step(i)
    for L in layers:
        st, det = moe.moe_check(L.ws)
        if st != moe.MOE_OK:
            raise RuntimeError(f"device error {moe.status_string(st)} ({det})")
    graphs = []
    n_graphs = max(n_copies, n_x)
    n0 = moe.moe_launch_total()
    for c in range(n_graphs):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            step(c)
        graphs.append(g)
    launches_per_step = (moe.moe_launch_total() - n0) // n_graphs
    for i in range(warmup):
        graphs[i % n_graphs].replay()
    torch.cuda.synchronize()

    # ---- timed region: exactly K steps (clocks sampled over a window around them)
    ms_total, clocks = timed_replays(lambda i: graphs[i % n_graphs].replay(), n_graphs, steps, stream, dev, world,
                                     args.clock_window)
    if cache_cfg:
        # the cache counters of the timed steps only: restart them and replay again
        cstats_t.zero_()
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev0.record(stream)
        for i in range(steps):
            graphs[i % n_graphs].replay()
        ev1.record(stream)
        torch.cuda.synchronize()
    ms_per_step = ms_total / steps
    value = whole_job_tokens_per_s(world, T, steps, ms_total)

    # ---- dominant kernel: the expert FFN stage, timed alone on the same stream
    # (route/select/permute outputs of each copy are already in place).
    # Decode: algorithmic bytes = weights of the distinct experts computed plus
    # the shared experts.  Prefill: algorithmic FLOPs = 2 * 3 * d * I per
    # computed (token, expert) row plus 2 * 3 * d * I_shared per token and
    # shared expert.
    fb, ff = [], []
    for c, L in enumerate(layers):
        off = bufs[c].expert_offsets.cpu().numpy()
        u = int((np.diff(off) > 0).sum())
        if cfg.keep_frac < 1.0:
            # FloE: dense up rows + gate/down rows of the union of kept channels
            moe.moe_expert_ffn(L.dims.with_T(T), xs[c], L.table, bufs[c].expert_offsets, bufs[c].perm,
                               cfg.keep_frac, bufs[c].y_perm, bufs[c].y_shared, L.ws, stream)
            torch.cuda.synchronize()
            ptr, words = moe.moe_floe_kept_mask(L.dims.with_T(T), L.ws)
            o = ptr - L.ws.data_ptr()
            kept = L.ws[o:o + int(off[-1]) * words * 4].view(torch.int32).cpu().numpy().view(np.uint32)
            kept = kept.reshape(-1, words)
            union_rows = 0
            for e in range(cfg.N):
                if off[e + 1] > off[e]:
                    union_rows += int(np.unpackbits(np.bitwise_or.reduce(kept[off[e]:off[e + 1]], axis=0)
                                                    .view(np.uint8)).sum())
            fb.append(u * cfg.I * cfg.d * esize + union_rows * 2 * cfg.d * esize + shared_bytes)
        else:
            fb.append(u * expert_bytes + shared_bytes)
        ff.append(6.0 * cfg.d * (int(off[-1]) * cfg.I + T * cfg.n_shared * cfg.I_shared))
    n_k = max(10 if phase == "prefill" else 50, min(2000, steps // 2))
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_k)]
    for i in range(n_k + n_copies):
        c = i % n_copies
        L, b = layers[c], bufs[c]
        D = L.dims.with_T(T)
        if i >= n_copies:
            evs[i - n_copies][0].record(stream)
        moe.moe_expert_ffn(D, xs[c], L.table, b.expert_offsets, b.perm, cfg.keep_frac, b.y_perm,
                           b.y_shared, L.ws, stream)
        if i >= n_copies:
            evs[i - n_copies][1].record(stream)
    torch.cuda.synchronize()
    k_ms = [a.elapsed_time(b) for a, b in evs]
    k_bytes = [fb[(i + n_copies) % n_copies] for i in range(n_k)]
    k_flops = [ff[(i + n_copies) % n_copies] for i in range(n_k)]
    path = moe.moe_expert_ffn_path(layers[0].dims.with_T(T), cfg.keep_frac)
    med_ms = statistics.median(k_ms)
    if phase == "decode":
        achieved = statistics.mean(k_bytes) / (med_ms / 1e3) / 1e9
        kname, ksrc = {
            "tc-decode": ("moe_expert_ffn (ffn_tcd_kernel + gemv_reduce_kernel)",
                          "ffn_tcd.cu"),
            "gemv-1tok": ("moe_expert_ffn (ffn_gemv1_kernel + gemv_reduce_kernel)", "ffn_gemv1.cu"),
            "gemv-floe": ("moe_expert_ffn (floe up/select/union/plan + sparse ffn_gemv_kernel"
                          " + gemv_reduce_kernel)", "ffn_gemv.cu"),
        }.get(path, ("moe_expert_ffn (ffn_gemv_kernel + gemv_reduce_kernel)", "ffn_gemv.cu"))
        roof = {"kernel": kname, "ffn_path": path, "bound": "hbm", "achieved": achieved, "unit": "GB/s",
                **fractions(achieved, hbm_gbs, NOMINAL_HBM_GBS, peak_src),
                "algorithmic_bytes_per_launch": float(statistics.mean(fb)), "median_launch_ms": med_ms,
                "avg_launch_ms": statistics.mean(k_ms), "launches_timed": n_k,
                "traffic": recorded_traffic(ksrc, wl_name)}
    else:
        # prefill: the bound is whichever roofline time is longer, the FLOPs at the
        # bf16 peak or the expert weight bytes at the HBM bandwidth (a short batch
        # of many experts, e.g. Granite-shaped at 1024 tokens, is HBM-bound)
        tflops = statistics.mean(k_flops) / (med_ms / 1e3) / 1e12
        gbs = statistics.mean(k_bytes) / (med_ms / 1e3) / 1e9
        t_flop = statistics.mean(ff) / (bf16_tflops * 1e12)
        t_byte = statistics.mean(fb) / (hbm_gbs * 1e9)
        pairs = T * cfg.k >= 256 * cfg.N  # the library's rule for the 2-CTA tiles
        common = {"kernel": "moe_expert_ffn (gather + ffn_tc_kernel%s: gate/up and down tiles in one launch)"
                            % ("<pairs> on CTA pairs, 2-CTA MMA" if pairs else "<single>"), "ffn_path": path}
        if t_byte > t_flop:
            roof = dict(common, bound="hbm", achieved=gbs, unit="GB/s",
                        **fractions(gbs, hbm_gbs, NOMINAL_HBM_GBS, peak_src), tensor_frac=tflops / bf16_tflops)
        else:
            sus, sus_src = sustained_bf16_tflops()
            roof = dict(common, bound="tensor", achieved=tflops, unit="TFLOP/s",
                        **fractions(tflops, bf16_tflops, NOMINAL_BF16_TFLOPS, peak_src + " bf16 burst"),
                        frac_of_sustained=tflops / sus, sustained_peak=sus, sustained_source=sus_src,
                        hbm_frac=gbs / hbm_gbs)
        roof.update({"algorithmic_flops_per_launch": float(statistics.mean(ff)),
                     "algorithmic_bytes_per_launch": float(statistics.mean(fb)),
                     "median_launch_ms": med_ms, "avg_launch_ms": statistics.mean(k_ms), "launches_timed": n_k,
                     "traffic": recorded_traffic("ffn_tc.cu", wl_name)})

    # the cache counters of the timed steps
    cache_info = None
    if cache_cfg:
        cs = cstats_t.cpu().numpy().astype(np.int64)
        steps_done = steps
        cache_info = {"capacity": capacity, "decay": decay, "start": f"experts 0..{capacity - 1}",
                      "hit_rate": float(cs[0]) / max(1, cs[1]), "miss_rate": 1.0 - float(cs[0]) / max(1, cs[1]),
                      "admitted_per_step": float(cs[2]) / steps_done, "evicted_per_step": float(cs[3]) / steps_done,
                      "stage_bytes_per_step": float(cs[2]) / steps_done * expert_bytes,
                      "note": "timed steps: layer (resident = cache, HYBRID misses) + cache update in CUDA "
                              "graphs; the pipeline and e2e loops also copy every admitted expert from pinned "
                              "host memory (moe_cache_step), overlapped with the following steps"}

    # ---- the look-ahead step alone, and what it predicted
    la_info = None
    if la_cfg:
        g_la = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_la, stream=stream):
            lookahead(0, xs[0])
        n_la = 200
        la_ev = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
        torch.cuda.synchronize()
        la_ev[0].record(stream)
        for _ in range(n_la):
            g_la.replay()
        la_ev[1].record(stream)
        torch.cuda.synchronize()
        la_us = la_ev[0].elapsed_time(la_ev[1]) * 1e3 / n_la
        # prediction quality over the distinct batches: the next layer's actual
        # routed sets (its router on x + this layer's output, through the same
        # entry point with tau = 0, one look-ahead layer) against the experts
        # predicted for it
        depths, confs, covered, routed_slots, staged = [], [], 0, 0, np.zeros(la_J)
        nxt_tok = torch.zeros((T, 1), dtype=torch.int64, device=dev)
        nxt_lay = torch.zeros(1, dtype=torch.int64, device=dev)
        nxt_logits = torch.zeros((1, T, cfg.N), dtype=torch.float32, device=dev)
        nxt_conf = torch.zeros((T, 1), dtype=torch.float32, device=dev)
        nxt_depth = torch.zeros(T, dtype=torch.int32, device=dev)
        for c in range(n_copies):
            forward(layers[c], bufs[c], xs[c], stream=stream)
            lookahead(c, xs[c])
            h1 = (xs[c].float() + bufs[c].out).to(base.dt).contiguous()
            moe.moe_prefetch_depth(layers[c].dims.with_T(T), h1, la_Wd[:1],
                                   None if la_bd is None else la_bd[:1], 0.0, 0, nxt_logits, nxt_conf, nxt_depth,
                                   nxt_tok, nxt_lay, layers[c].ws, stream)
            torch.cuda.synchronize()
            depths += la_depth.cpu().tolist()
            confs.append(la_conf.double().cpu().numpy())
            pred = int(la_lay[0].item()) & ((1 << 64) - 1)
            for t in range(T):
                actual = int(nxt_tok[t, 0].item()) & ((1 << 64) - 1)
                covered += bin(actual & pred).count("1")
                routed_slots += cfg.k
            staged += [bin(int(v) & ((1 << 64) - 1)).count("1") for v in la_lay.cpu().tolist()]
        la_info = {"look_ahead_layers": la_J, "tau": la_tau, "d_min": la_dmin,
                   "us_per_call": la_us, "launches_per_call": la_J + 1,
                   "mean_depth": float(np.mean(depths)),
                   "depth_histogram": np.bincount(np.asarray(depths), minlength=la_J + 1).tolist(),
                   "mean_confidence_per_layer": np.concatenate(confs).mean(axis=0).round(4).tolist(),
                   "experts_to_stage_per_layer": (staged / n_copies).round(2).tolist(),
                   "next_layer_coverage": covered / routed_slots,
                   "note": "draft head = the look-ahead routers on the current hidden state; coverage = "
                           "routed slots of the next layer (its router on x + this layer's output) whose "
                           "expert was predicted for it"}

    # ---- end to end through the public API: pinned host x -> device, layer
    # forward, result -> pinned host, every step
    x_host = [xs[c].cpu().pin_memory() for c in range(n_x)]
    out_host = [torch.empty_like(bufs[c].out, device="cpu").pin_memory() for c in range(n_copies)]
    n_e2e = max(5 if phase == "prefill" else 20, min(steps, 1000))
    if cache_cfg:
        # the overlapped pipeline: admissions copied on a staging stream while
        # later steps run on the experts already landed (one layer copy)
        from expert_routing_ffn_gb300.layer import CachePipeline
        pipe = CachePipeline(layers[0], capacity, decay, stream=stream)
        pipe.start((1 << capacity) - 1)
        for i in range(max(3, warmup)):
            pipe.step(bufs[0], xs[i % n_x], n_resident=0)
        stream.synchronize()
        # steps back to back (the host never waits on the step path)
        n_pipe = max(50, min(steps, 2000))
        s0 = pipe.pipe.staged_bytes
        t0 = time.perf_counter()
        for i in range(n_pipe):
            pipe.step(bufs[0], xs[i % n_x], n_resident=0)
        stream.synchronize()
        pipe_s = time.perf_counter() - t0
        cache_info["pipeline"] = {"tokens_per_s": world * T * n_pipe / max_over_ranks(world, pipe_s),
                                  "us_per_step": 1e6 * pipe_s / n_pipe, "steps": n_pipe,
                                  "staged_bytes_per_step": (pipe.pipe.staged_bytes - s0) / n_pipe,
                                  "note": "moe_cache_step back to back: layer on cache & landed, heat/cache "
                                          "update, admissions copied on a staging stream; host clock"}
        s0 = pipe.pipe.staged_bytes
    plain = not la_cfg and not cache_cfg
    if plain:
        # moe_layer_forward_host: copy in, layer, copy out as one replayed
        # graph per (layer copy, input buffer); captured here, before timing
        for i in range(max(n_copies, n_x)):
            forward_host(layers[i % n_copies], bufs[i % n_copies], xs[i % n_x], x_host[i % n_x],
                         out_host[i % n_copies], stream=stream)
        stream.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(n_e2e):
        c = 0 if cache_cfg else i % n_copies
        xc = xs[i % n_x]
        if plain:
            forward_host(layers[c], bufs[c], xc, x_host[i % n_x], out_host[c], stream=stream)
            stream.synchronize()
            continue
        xc.copy_(x_host[i % n_x], non_blocking=True)
        if la_cfg:
            forward(layers[c], bufs[c], xc, stream=stream)
            lookahead(c, xc)
        else:
            pipe.step(bufs[0], xc, n_resident=0)
        out_host[c].copy_(bufs[c].out, non_blocking=True)
        stream.synchronize()
    torch.cuda.synchronize()
    e2e_s = max_over_ranks(world, time.perf_counter() - t0)
    e2e_value = world * T * n_e2e / e2e_s
    if cache_cfg:
        cache_info["e2e_staged_bytes_per_step"] = (pipe.pipe.staged_bytes - s0) / n_e2e
        pipe.drain()

    # ---- expert staging over the host link (EXACT-mode fetches): copy every
    # expert of one layer copy from pinned host memory with moe_stage_experts
    n_stage = min(cfg.N, 8)
    host_w = [[layers[0].w_gate[e].cpu().pin_memory() for e in range(cfg.N)],
              [layers[0].w_up[e].cpu().pin_memory() for e in range(cfg.N)],
              [layers[0].w_down[e].cpu().pin_memory() for e in range(cfg.N)]]
    side = torch.cuda.Stream(device=dev)
    done = torch.cuda.Event()
    mask = (1 << n_stage) - 1
    D1 = layers[0].dims.with_T(T)
    moe.moe_stage_experts(D1, mask, *host_w, list(layers[0].w_gate), list(layers[0].w_up),
                          list(layers[0].w_down), side, done)
    side.synchronize()
    t0 = time.perf_counter()
    reps = 3
    for _ in range(reps):
        nbytes = moe.moe_stage_experts(D1, mask, *host_w, list(layers[0].w_gate), list(layers[0].w_up),
                                       list(layers[0].w_down), side, done)
    side.synchronize()
    stage_s = time.perf_counter() - t0
    staging = {"gbps": reps * nbytes / stage_s / 1e9, "bytes_per_call": nbytes,
               "experts_per_call": n_stage, "note": "pinned host -> HBM, cudaMemcpyAsync on a side stream"}

    # ---- routing statistics of the last layer forward of each copy (the
    # counters of moe_select_resident: hit / substitute / LoRE / fetch slots,
    # overlap of the routed set with the prefetch set, mean delta_hat, delta*)
    torch.cuda.synchronize()
    cnt = np.zeros(moe.MOE_NUM_COUNTERS, np.int64)
    for c in range(n_copies):
        cnt += bufs[c].counters.cpu().numpy().astype(np.int64)
    toks = n_copies * T
    routing = {"tokens": toks, "slots": toks * cfg.k,
               "hit": int(cnt[0]), "substitute": int(cnt[1]), "lore": int(cnt[2]), "fetch": int(cnt[3]),
               "shortfall_tokens": int(cnt[7]),
               # counted only when the prefetch set takes part in the selection
               "overlap_rate": float(cnt[4]) / toks if cfg.use_prefetch_mask else None,
               "mean_delta_hat": float(cnt[5]) / toks, "mean_delta_star": float(cnt[6]) / toks,
               "tau": cfg.tau, "gamma": cfg.gamma}

    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": steps, "warmup": warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": cfg.wtype if cfg.wtype == "bf16" else "f32",
        "data": "synthetic (seeded N(0,0.02^2) weights, N(0,1) tokens; shapes of the named model)",
        "config": {"workload": wl_name, "tokens_per_step": T, "d": cfg.d, "experts": cfg.N,
                   "top_k": cfg.k, "intermediate": cfg.I, "shared_experts": cfg.n_shared,
                   "floe_keep_frac": cfg.keep_frac,
                   "miss_policy": ["exact", "substitute", "lore", "hybrid"][cfg.policy],
                   "resident": cfg.n_resident, "parallelism": f"replicas x{world}",
                   "l2": f"inputs larger than L2: {n_copies} rotating layer copies of "
                         f"{layer_bytes / 1e9:.2f} GB", "cuda_graph": True},
        "roofline": roof,
        "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": xs[0].numel() * xs[0].element_size(),
                "d2h_bytes_per_step": bufs[0].out.numel() * 4, "steps": n_e2e,
                "note": "moe_layer_forward_host per step (pinned x in, layer, out to pinned memory, replayed "
                        "as one CUDA graph by the library) and a stream sync"},
        "gpu_launches": int(launches_per_step * steps),
        "staging": staging,
        "routing": routing,
        "clocks": clocks,
    }
    if la_info:
        # SPICE's minimum depth for one expert of this layer, at the measured
        # layer step time, over a PCIe 4.0 x16 link and over this box's
        # measured host link
        step_s = ms_per_step / 1e3
        la_info["d_min_formula"] = {
            "expert_bytes": expert_bytes, "layer_us": ms_per_step * 1e3,
            "pcie4_x16": moe.moe_prefetch_min_depth(expert_bytes, PCIE4_X16_BYTES_PER_S, step_s),
            "measured_host_link": moe.moe_prefetch_min_depth(expert_bytes, staging["gbps"] * 1e9, step_s)}
        line["lookahead"] = la_info
        line["config"]["lookahead"] = f"{la_J} layers, tau {la_tau}, d_min {la_dmin}"
    if cache_info:
        line["config"]["resident"] = f"expert cache of {capacity} (heat decay {decay})"
        line["e2e"]["h2d_bytes_per_step"] += cache_info["e2e_staged_bytes_per_step"]
        line["e2e"]["d2h_bytes_per_step"] += 32
        line["e2e"]["note"] = "moe_cache_step per step (layer, cache update, admissions copied on a staging " \
                              "stream) with pinned-host copies of x and out and a stream sync"
        line["cache"] = cache_info
    # the whole step against the same bound: the FFN's algorithmic work plus
    # the router and prefetch-router weights (decode) or FLOPs (prefill)
    router_bytes = 2 * cfg.N * cfg.d * esize + 4 * cfg.d
    if roof["bound"] == "hbm":
        work = float(statistics.mean(fb)) + router_bytes
        ach = work / (ms_per_step / 1e3) / 1e9
        line["layer_roofline"] = {"bound": "hbm", "bytes_per_step": work, "achieved": ach, "unit": "GB/s",
                                  **fractions(ach, hbm_gbs, NOMINAL_HBM_GBS, peak_src)}
    else:
        work = float(statistics.mean(ff)) + 2.0 * T * 2 * cfg.N * cfg.d
        ach = work / (ms_per_step / 1e3) / 1e12
        # the whole step is timed inside a long loop: the sustained rate is its denominator
        sus, sus_src = sustained_bf16_tflops()
        line["layer_roofline"] = {"bound": "tensor", "flops_per_step": work, "achieved": ach, "unit": "TFLOP/s",
                                  **fractions(ach, sus, NOMINAL_BF16_TFLOPS, sus_src),
                                  "frac_of_burst": ach / bf16_tflops}
    if rank == 0 and with_cpu and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(cfg, W, T, args.cpu_seconds, wl_name=wl_name)
    del layers, bufs, base
    return line


def main():
    args = parse()
    wl_name = args.workload
    both = wl_name == DEFAULT_WORKLOAD and not args.no_prefill
    if args.impl == "reference":
        run_reference(args, wl_name, int(os.environ.get("RANK", "0")), both)
        return

    import torch
    import expert_routing_ffn_gb300 as moe

    world, rank, local = dist_setup(args.gpus)
    dev = torch.device("cuda", local if world > 1 else 0)
    moe.lib()  # fails loudly if the CUDA library is missing
    line = run_workload(args, wl_name, world, rank, dev, args.steps, args.warmup)
    if both:
        # the prefill half of the metric: the largest single-GPU layer shape,
        # its own timed steps, roofline, end-to-end figure and CPU baseline
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        pf = run_workload(args, PREFILL_WORKLOAD, world, rank, dev, max(10, min(args.steps, 100)),
                          max(3, min(args.warmup, 5)))
        line["prefill"] = nested(pf)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
