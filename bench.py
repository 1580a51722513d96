#!/usr/bin/env python
"""Throughput of the fused MoE-LoRA expert layer on GB300; prints one JSON line.

A step is one call of the whole layer (route, align, gather, gate_up GEMM,
gate_up shrink, expand + SwiGLU, down GEMM, down shrink, expand + combine) on
one batch of the GPT-OSS-20B-shaped decode workload (T = 64 tokens, one per
request, hidden 2880, intermediate 2880, 32 experts top-4, 8 adapters r = 32),
with seeded synthetic inputs and random weights.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun each rank drives its own GPU with an independent replica of the
layer (the layer has no exchange step); the elapsed time is the maximum over
ranks and the value counts the tokens of all ranks. ``--impl reference`` times
the fp64 CPU oracle on the host cores instead (rank 0 only).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "MoE-LoRA layer tokens/s; shrink/expand HBM GB/s as % of ~8 TB/s peak"
UNIT = "tokens/s"
DEFAULT_WORKLOAD = "gptoss20b_decode"
STAGES = ["route", "align", "gather", "gate_up_gemm", "gate_up_shrink", "gate_up_expand_swiglu",
          "down_gemm", "down_shrink", "down_expand_combine"]


# ----------------------------------------------------------------------------
# ranks
# ----------------------------------------------------------------------------
def world():
    return (int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")),
            int(os.environ.get("LOCAL_RANK", "0")))


def combine_ranks(elapsed_s: float, units: float):
    """(max elapsed over ranks, sum of units over ranks); plain values at world size 1."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return elapsed_s, units
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([elapsed_s], dtype=torch.float64, device=dev)
    u = torch.tensor([units], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


# ----------------------------------------------------------------------------
# algorithmic bytes / flops per launch (the minimum data each stage must move)
# ----------------------------------------------------------------------------
# Stage names in the order of the layer's event marks ([0] .. [8]); the fused chain
# (expand inside the grouped GEMMs) has an empty slot where the SwiGLU expand was.
FUSED_STAGES = ["route", "align", "gather", "gate_up_shrink", "gate_up_gemm_expand_swiglu", None,
                "down_shrink", "down_gemm_expand", "combine"]


def chain_stages(fused: bool):
    return FUSED_STAGES if fused else STAGES


def workload_stats(ids, token_adapter, E: int):
    """Counts that set the algorithmic traffic: touched experts, (e, l) pairs, rows."""
    import numpy as np
    ids = np.asarray(ids)
    ad = np.asarray(token_adapter)
    T, k = ids.shape
    e_touched = len(np.unique(ids))
    lora_tok = ad >= 0
    pairs = set()
    for t in range(T):
        if ad[t] >= 0:
            for j in range(k):
                pairs.add((int(ids[t, j]), int(ad[t])))
    return dict(T=T, k=k, S=T * k, E_touched=e_touched, P=len(pairs),
                T_L=int(lora_tok.sum()), S_L=int(lora_tok.sum()) * k)


def stage_bytes(st: dict, H: int, I: int, E: int, r: int, fused: bool = False) -> dict:
    """Minimum bytes each stage reads + writes (bf16 = 2, fp32/int32 = 4). z is fp32 by
    slot in the unfused chain and a bf16 pair (4 bytes) by sorted row in the fused one."""
    S, T, S_L, T_L, P, Et = st["S"], st["T"], st["S_L"], st["T_L"], st["P"], st["E_touched"]
    common = {
        "route": T * E * 4 + S * 8,
        "align": S * 4 + T * 4 + S * 16,
        "gather": T * H * 2 + S * H * 2,
        "gate_up_shrink": P * r * H * 2 + T_L * H * 2 + S_L * r * 4,
        "down_shrink": P * r * I * 2 + S_L * I * 2 + S_L * r * 4,
    }
    if fused:
        common.update({
            # W1, gathered rows, B1, z in; h out
            "gate_up_gemm_expand_swiglu": Et * 2 * I * H * 2 + S * H * 2 + P * 2 * I * r * 2
            + S_L * r * 4 + S * I * 2,
            # W2, h rows, B2, z in; fp32 rows out
            "down_gemm_expand": Et * H * I * 2 + S * I * 2 + P * H * r * 2 + S_L * r * 4
            + S * H * 4,
            "combine": S * H * 4 + S * 8 + T * H * 2,
        })
        return common
    common.update({
        "gate_up_gemm": Et * 2 * I * H * 2 + S * H * 2 + S * 2 * I * 4,
        "gate_up_expand_swiglu": P * 2 * I * r * 2 + S_L * r * 4 + S * 2 * I * 4 + S * I * 2,
        "down_gemm": Et * H * I * 2 + S * I * 2 + S * H * 4,
        "down_expand_combine": P * H * r * 2 + S_L * r * 4 + 2 * S_L * H * 4 + S * H * 4
        + S * 4 + T * H * 2,
    })
    return common


def stage_flops(st: dict, H: int, I: int, r: int, fused: bool = False) -> dict:
    S, S_L = st["S"], st["S_L"]
    f = {"gate_up_shrink": 2 * S_L * r * H, "down_shrink": 2 * S_L * r * I}
    if fused:
        f["gate_up_gemm_expand_swiglu"] = 2 * S * 2 * I * H + 2 * S_L * 2 * I * r
        f["down_gemm_expand"] = 2 * S * H * I + 2 * S_L * H * r
        return f
    f.update({"gate_up_gemm": 2 * S * 2 * I * H, "down_gemm": 2 * S * H * I,
              "gate_up_expand_swiglu": 2 * S_L * 2 * I * r, "down_expand_combine": 2 * S_L * H * r})
    return f


GEMM_STAGES = ("gate_up_gemm", "down_gemm", "gate_up_gemm_expand_swiglu", "down_gemm_expand")


# ----------------------------------------------------------------------------
# clocks during the timed region (read only: NVML queries, or nvidia-smi)
# ----------------------------------------------------------------------------
class NvmlClock:
    """The GPU's SM clock, power and clock-event reasons, read through NVML every
    millisecond on a thread while started. Reading only: nothing is set."""
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, local_rank: int):
        import ctypes
        self.ok = False
        self.samples = []
        self._thread = None
        self._stop = threading.Event()
        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
        except OSError:
            return
        if nv.nvmlInit_v2() != 0:
            return
        h = ctypes.c_void_p()
        rc = 1
        bus = pci_bus_id(local_rank)
        if bus:
            rc = nv.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), ctypes.byref(h))
        if rc != 0:
            rc = nv.nvmlDeviceGetHandleByIndex_v2(int(gpu_index_for_smi(local_rank)),
                                                   ctypes.byref(h))
        if rc != 0:
            return
        self.ct, self.nv, self.h = ctypes, nv, h
        mx = ctypes.c_uint(0)
        nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx))  # 1: the SM clock
        self.max_mhz = mx.value
        self._reasons = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(nv, "nvmlDeviceGetCurrentClocksThrottleReasons")
        self.ok = True

    def read(self):
        ct, nv, h = self.ct, self.nv, self.h
        c, p, r = ct.c_uint(0), ct.c_uint(0), ct.c_ulonglong(0)
        nv.nvmlDeviceGetClockInfo(h, 1, ct.byref(c))
        nv.nvmlDeviceGetPowerUsage(h, ct.byref(p))
        self._reasons(h, ct.byref(r))
        return time.time(), c.value, p.value / 1000.0, r.value

    def _run(self):
        while not self._stop.is_set():
            self.samples.append(self.read())
            time.sleep(0.001)

    def start(self):
        if self.ok:
            self._thread = threading.Thread(target=self._run, daemon=True)
            self._thread.start()
            t0 = time.time()
            while not self.samples and time.time() - t0 < 2.0:
                time.sleep(0.001)

    def stop(self):
        self._stop.set()
        if self._thread is not None:
            self._thread.join(timeout=2)

    def summary(self, t0: float, t1: float):
        if not self.ok:
            return None
        win = [s for s in self.samples if t0 <= s[0] <= t1]
        note = None
        if not win and self.samples:
            mid = 0.5 * (t0 + t1)
            win = [min(self.samples, key=lambda s: abs(s[0] - mid))]
            note = "timed region shorter than one sample; nearest sample used"
        reasons = set()
        for s in win:
            for bit, name in self.REASONS.items():
                if s[3] & bit:
                    reasons.add(name)
        after = self.read()
        out = {"sm_mhz": statistics.median(s[1] for s in win) if win else None,
               "sm_max_mhz": self.max_mhz, "reasons": sorted(reasons), "samples": len(win),
               "power_w_max": max((s[2] for s in win), default=None), "source": "nvml, 1 ms",
               "after_timed": {"sm_mhz": after[1],
                               "reasons": sorted(n for b, n in self.REASONS.items() if after[3] & b)}}
        if note:
            out["note"] = note
        return out


def pci_bus_id(local_rank: int):
    """NVML's PCI bus id string of torch's device local_rank, or None."""
    try:
        import torch
        p = torch.cuda.get_device_properties(local_rank)
        return f"{p.pci_domain_id:08x}:{p.pci_bus_id:02x}:{p.pci_device_id:02x}.0"
    except Exception:  # attributes absent in this torch build
        return None


def gpu_index_for_smi(local_rank: int) -> str:
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        parts = [p.strip() for p in vis.split(",") if p.strip()]
        if local_rank < len(parts):
            return parts[local_rank]
    return str(local_rank)


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


STAGE_SOURCES = {
    "route": ["route.cu"], "align": ["align.cu"], "gather": ["grouped_gemm.cu"],
    "gate_up_gemm": ["grouped_gemm.cu"], "down_gemm": ["grouped_gemm.cu"],
    "gate_up_shrink": ["lora_shrink.cu"], "down_shrink": ["lora_shrink.cu"],
    "gate_up_expand_swiglu": ["lora_expand.cu"], "down_expand_combine": ["lora_expand.cu"],
    "gate_up_gemm_expand_swiglu": ["fused_gemm.cu"], "down_gemm_expand": ["fused_gemm.cu"],
    "combine": ["lora_expand.cu"],
}


def source_hash(stage: str) -> str:
    import hashlib
    csrc = os.path.join(ROOT, "expert_adapter_gemms_gb300", "csrc")
    h = hashlib.sha256()
    for f in STAGE_SOURCES.get(stage, []) + ["common.cuh"]:
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(stage: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, or None when there is no
    capture for this stage and workload or the kernel's source changed since."""
    p = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        for line in f:
            parts = line.split()
            if line.startswith("#") or len(parts) < 4:
                continue
            if parts[0] == stage and parts[1] == workload:
                return float(parts[2]) if parts[3] == source_hash(stage) else None
    return None


# ----------------------------------------------------------------------------
# CPU oracle timing (the baseline leg and the reference arm)
# ----------------------------------------------------------------------------
class OracleStep:
    """One step of the fp64 CPU oracle on the first `tokens` tokens of a batch.
    Weights are converted to fp64 once, before any timing (conversion excluded)."""

    def __init__(self, inp, tokens=None):
        import oracle
        self.oracle = oracle
        self.inp = inp
        self.n = inp.T if tokens is None else max(1, min(inp.T, int(tokens)))
        self.W = {n: oracle.as_f64(getattr(inp, n)) for n in ("W1", "W2", "A1", "B1", "A2", "B2")
                  if getattr(inp, n) is not None}
        self.x = oracle.as_f64(inp.x)[: self.n]
        self.logits = inp.logits.numpy()[: self.n]
        self.ad = inp.token_adapter.numpy()[: self.n]

    def __call__(self):
        o, W = self.oracle, self.W
        ids, w = o.route_topk_softmax(self.logits, self.inp.k)
        return o.moe_lora_layer(self.x, W["W1"], W["W2"], ids, w, self.ad, W.get("A1"),
                                W.get("B1"), W.get("A2"), W.get("B2"))


def cpu_oracle_rate(inp, seconds: float, max_reps: int = 1000):
    """Tokens/s of the fp64 oracle on this host: whole batches until `seconds` pass."""
    step = OracleStep(inp)
    t0 = time.perf_counter()
    reps = 0
    while True:
        step()
        reps += 1
        el = time.perf_counter() - t0
        if el >= seconds or reps >= max_reps:
            break
    return inp.T * reps / el, reps, el


def cpu_cores():
    try:
        n = len(os.sched_getaffinity(0))
    except AttributeError:
        n = os.cpu_count() or 1
    for v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        if os.environ.get(v, "").isdigit():
            n = min(n, int(os.environ[v]))
    return n


def host_info() -> dict:
    """CPU model and BLAS thread pool of the host the oracle runs on (best effort: a field
    that cannot be read is reported as unknown, never an error)."""
    import platform
    import subprocess
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.split(":")[0].strip() == "Model name":
                model = line.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    if not model:
        try:
            with open("/proc/cpuinfo") as f:
                for line in f:
                    if line.startswith("model name"):
                        model = line.split(":", 1)[1].strip()
                        break
        except OSError:
            pass
    blas = None
    try:
        import numpy  # noqa: F401  (loads the BLAS library the oracle uses)
        from threadpoolctl import threadpool_info
        pools = [p for p in threadpool_info() if p.get("user_api") == "blas"]
        if pools:
            blas = {"library": pools[0].get("internal_api"), "threads": pools[0].get("num_threads")}
    except Exception:  # threadpoolctl absent or unable to inspect the loaded libraries
        pass
    if blas is None:
        env = {v: os.environ[v] for v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS",
                                           "MKL_NUM_THREADS") if v in os.environ}
        blas = {"library": "unknown", "threads": env or "library default"}
    return {"cpu_model": model or platform.processor() or platform.machine(), "blas": blas}


# ----------------------------------------------------------------------------
# arms
# ----------------------------------------------------------------------------
def workload_config(inp, extra=None):
    c = {"workload": inp.name, "T": inp.T, "H": inp.H, "I": inp.I, "E": inp.E, "k": inp.k,
         "L": inp.L, "r": inp.r, "weights": "random N(0,0.02) bf16", "x": "N(0,1) bf16"}
    if extra:
        c.update(extra)
    return c


def run_reference(args):
    """The oracle as the reference arm: exactly `steps` timed steps after `warmup`, each on
    a token sample sized so the whole run stays within --ref-budget-s."""
    nw, rank, _ = world()
    if rank != 0:
        return 0
    from workloads import make_workload_inputs
    inp = make_workload_inputs(args.workload)
    full = OracleStep(inp)
    t0 = time.perf_counter()
    full()
    t_full = time.perf_counter() - t0
    per_step = args.ref_budget_s / max(1, args.steps + args.warmup)
    n = inp.T if t_full <= per_step else max(1, int(inp.T * per_step / t_full))
    step = full if n == inp.T else OracleStep(inp, n)
    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    el = time.perf_counter() - t0
    rate = step.n * args.steps / el
    line = {"metric": METRIC, "value": rate, "unit": UNIT, "impl": "reference", "n_gpus": nw,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * el / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": workload_config(inp, {"parallelism": f"replicas x{nw}" if nw > 1
                                            else "single device"}),
            "cpu_baseline": {"value": rate, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
                             "sample": f"{step.n} of {inp.T} tokens per step (fp64 NumPy oracle)",
                             **host_info()},
            "e2e": {"value": rate, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def launches_per_layer(m, inp) -> int:
    """Kernels one layer call launches (routed from logits), as the library plans it."""
    return m.moe_lora_layer_plan(inp.T, inp.k, inp.E, inp.L, inp.H, inp.I, inp.r)["launches"]


def multi_layer(m, inp, W1, W2, lora, lg_d, ta_d, x_d, ws, n_layers, steps, warmup):
    """N layers chained on one stream, layer i + 1 reading layer i's y, timed eagerly and
    replayed from one CUDA graph. Layer i's weights, adapters and router logits are layer
    0's rolled by i along the expert axis: the same statistics in distinct memory, so every
    layer streams its own weights from HBM. Programmatic dependent launch chains the
    kernels across layer boundaries as within a layer."""
    import torch
    layers = []
    for i in range(n_layers):
        if i == 0:
            layers.append((W1, W2, lora, lg_d))
        else:
            layers.append((torch.roll(W1, i, 0), torch.roll(W2, i, 0),
                           {kk: torch.roll(v, i, 1) for kk, v in lora.items()},
                           torch.roll(lg_d, i, 1)))
    ys = [torch.empty_like(x_d) for _ in range(n_layers)]

    def run():
        xin = x_d
        for (w1, w2, lo, lg), y in zip(layers, ys):
            m.moe_lora_layer(xin, w1, w2, logits=lg, k=inp.k, token_adapter=ta_d, y=y,
                             workspace=ws, **lo)
            xin = y

    def timed(fn):
        for _ in range(warmup):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(steps):
            fn()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) * 1e3 / steps  # us per pass over all layers

    eager_us = timed(run)
    y_eager = ys[-1].clone()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        run()  # warm-up on the capture stream
    torch.cuda.current_stream().wait_stream(side)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        run()
    graph_us = timed(g.replay)
    same = bool(torch.equal(ys[-1], y_eager))
    err = m.get_error(ws)
    del g, layers, ys
    return {"layers": n_layers, "steps": steps,
            "eager_us_per_layer": round(eager_us / n_layers, 2),
            "graph_us_per_layer": round(graph_us / n_layers, 2),
            "graph_tokens_s": inp.T * n_layers / (graph_us * 1e-6),
            "graph_matches_eager": same, "device_error": err}


class Layer:
    """One workload's inputs on the device and a layer call over them."""

    def __init__(self, m, name, expand_mode=0):
        import torch
        from workloads import make_workload_inputs
        self.m = m
        self.expand_mode = expand_mode
        self.inp = inp = make_workload_inputs(name)
        d = lambda t: None if t is None else t.to("cuda").contiguous()  # noqa: E731
        self.W1, self.W2 = d(inp.W1), d(inp.W2)
        self.lora = dict(A1=d(inp.A1), B1=d(inp.B1), A2=d(inp.A2), B2=d(inp.B2)) if inp.L else {}
        self.x, self.lg, self.ta = d(inp.x), d(inp.logits), d(inp.token_adapter)
        self.y = torch.empty((inp.T, inp.H), dtype=torch.bfloat16, device="cuda")
        self.ws = m.new_workspace(inp.T, inp.k, inp.E, inp.L, inp.H, inp.I, inp.r)
        self.plan = m.moe_lora_layer_plan(inp.T, inp.k, inp.E, inp.L, inp.H, inp.I, inp.r,
                                          expand_mode=expand_mode)

    def __call__(self, events=None, adapters=True):
        inp = self.inp
        if adapters:
            self.m.moe_lora_layer(self.x, self.W1, self.W2, logits=self.lg, k=inp.k,
                                  token_adapter=self.ta, y=self.y, workspace=self.ws,
                                  events=events, expand_mode=self.expand_mode, **self.lora)
        else:  # the base MoE alone (L = 0): the same layer without adapters
            self.m.moe_lora_layer(self.x, self.W1, self.W2, logits=self.lg, k=inp.k, y=self.y,
                                  workspace=self.ws, events=events, expand_mode=self.expand_mode)


def timed_steps(fn, steps, stream):
    """Seconds for `steps` calls of fn on `stream`, by CUDA events recorded on it."""
    import torch
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        fn()
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / 1e3


def stage_table(layer, kernel_steps, stream, peaks):
    """Per-stage CUDA-event durations (a separate instrumented pass with events between the
    launches) against each stage's algorithmic bytes and flops."""
    import numpy as np
    import torch
    inp, fused = layer.inp, bool(layer.plan["fused_expand"])
    names = chain_stages(fused)
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(len(names) + 1)]
    for ev in evs:  # torch creates CUDA events lazily, on first record
        ev.record(stream)
    torch.cuda.synchronize()
    acc = [0.0] * len(names)
    for _ in range(kernel_steps):
        layer(events=evs)
        torch.cuda.synchronize()
        for i in range(len(names)):
            acc[i] += evs[i].elapsed_time(evs[i + 1])
    ids = torch.topk(inp.logits, inp.k, dim=1).indices.numpy()  # accounting only
    st = workload_stats(ids, inp.token_adapter.numpy() if inp.L else np.full(inp.T, -1), inp.E)
    sb = stage_bytes(st, inp.H, inp.I, inp.E, inp.r, fused)
    sf = stage_flops(st, inp.H, inp.I, inp.r, fused)
    hbm = float(peaks["hbm_gbs"])
    tflops = float(peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"]))
    kernels = {}
    for name, a in zip(names, acc):
        if name is None:
            continue
        ms = a / kernel_steps
        gbs = sb[name] / (ms * 1e-3) / 1e9 if ms > 0 else None
        k = {"us": round(ms * 1e3, 2), "alg_bytes": int(sb[name]),
             "GB_s": round(gbs, 1) if gbs else None,
             "hbm_frac": round(gbs / hbm, 3) if gbs else None}
        if name in sf and ms > 0:
            k["TFLOP_s"] = round(sf[name] / (ms * 1e-3) / 1e12, 2)
            if name in GEMM_STAGES:
                k["tensor_frac_of_sustained"] = round(k["TFLOP_s"] / tflops, 3)
        kernels[name] = k
    return kernels, sb


def stream_floor(stream, sizes_mb=(29.7, 66.0, 300.0), reps=16):
    """The time of one launch that reads and writes a given number of bytes, by CUDA events
    over `reps` back-to-back device-to-device copies (torch's copy kernel) through rotating
    buffers larger than L2. A short stream carries a fixed cost (launch, ramp-up of the
    memory pipeline, drain) that no kernel design removes; these figures put the roofline
    fractions of the decode LoRA kernels (30-66 MB each) in context."""
    import torch
    out = {}
    for mb in sizes_mb:
        n = int(mb * 1e6 / 2) // 2 * 2  # bf16 elements moved: half read, half written
        half = n // 2
        nbuf = max(2, int(512e6 // (n * 2)) + 1)  # > 512 MB in rotation: no L2 reuse
        src = [torch.empty(half, dtype=torch.bfloat16, device="cuda") for _ in range(nbuf)]
        dst = [torch.empty(half, dtype=torch.bfloat16, device="cuda") for _ in range(nbuf)]
        for i in range(nbuf):
            dst[i].copy_(src[i])
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(reps):
            dst[i % nbuf].copy_(src[i % nbuf])
        e1.record(stream)
        torch.cuda.synchronize()
        us = e0.elapsed_time(e1) * 1e3 / reps
        out[f"{mb:g}MB"] = {"us": round(us, 2), "GB_s": round(2 * half * 2 / (us * 1e-6) / 1e9, 1)}
        del src, dst
        torch.cuda.empty_cache()
    return out


def measure(layer, steps, warmup, kernel_steps, stream, peaks):
    """ms per step (CUDA events over exactly `steps` calls after `warmup`), the base MoE
    alone for the marginal cost of the adapters, and the per-stage table."""
    import torch
    for _ in range(warmup):
        layer()
    torch.cuda.synchronize()
    el = timed_steps(layer, steps, stream)
    out = {"tokens_s": layer.inp.T * steps / el, "ms_per_step": 1e3 * el / steps,
           "fused_expand": layer.plan["fused_expand"], "launches": layer.plan["launches"]}
    if layer.inp.L:
        for _ in range(warmup):
            layer(adapters=False)
        torch.cuda.synchronize()
        base = timed_steps(lambda: layer(adapters=False), steps, stream)
        out["base_moe_ms_per_step"] = 1e3 * base / steps
        out["lora_marginal_us"] = round(1e6 * (el - base) / steps, 2)
    out["kernels"], _ = stage_table(layer, kernel_steps, stream, peaks)
    if layer.m.get_error(layer.ws):
        raise RuntimeError(f"device error word set on {layer.inp.name}")
    return out


def run_ours(args):
    import torch
    import torch.distributed as dist

    nw, rank, local = world()
    if nw > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    import expert_adapter_gemms_gb300 as m

    layer = Layer(m, args.workload, args.expand_mode)
    inp = layer.inp
    stream = torch.cuda.current_stream()
    peaks, peak_kind = measured_peaks()

    clocks = NvmlClock(local)
    clocks.start()  # returns once the first sample is in
    for _ in range(args.warmup):
        layer()
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    t0 = time.time()
    el_s = timed_steps(layer, args.steps, stream)
    t1 = time.time()
    barrier()
    el_max, tokens_all = combine_ranks(el_s, inp.T * args.steps)
    value = tokens_all / el_max
    clk = clocks.summary(t0, t1)
    clocks.stop()
    if clk is None:
        clk = {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["NVML unavailable"], "samples": 0}
    err = m.get_error(layer.ws)
    if err:
        raise RuntimeError(f"device error word {err:#x} after the timed steps")

    # end to end through the host-staged C-ABI call: every step copies its inputs (x, logits,
    # adapter ids) from one page-locked host block and reads y back into host memory
    io = m.new_host_io(inp.T, inp.H, inp.E, with_adapter=inp.L > 0)
    io.x.copy_(inp.x)
    io.logits.copy_(inp.logits)
    if io.token_adapter is not None:
        io.token_adapter.copy_(inp.token_adapter)
    h2d = io.in_bytes
    d2h = io.y_host.numel() * io.y_host.element_size()

    def e2e_step():
        m.moe_lora_layer_host(io, layer.W1, layer.W2, k=inp.k, workspace=layer.ws,
                              expand_mode=args.expand_mode, **layer.lora)

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize()
    barrier()
    e2e_max, e2e_tokens = combine_ranks(timed_steps(e2e_step, args.steps, stream),
                                        inp.T * args.steps)
    if not torch.equal(io.y_host, layer.y.cpu()):
        raise RuntimeError("the host-staged step's y differs from the device-pointer call's")

    # per stage, and the base MoE alone
    head = measure(layer, max(args.steps, 20), 3, args.kernel_steps, stream, peaks)
    kernels = head["kernels"]
    dname = max(kernels, key=lambda n: kernels[n]["us"])
    dk = kernels[dname]
    hbm = float(peaks["hbm_gbs"])
    achieved = dk["alg_bytes"] / (dk["us"] * 1e-6) / 1e9
    roof = {"kernel": dname, "bound": "hbm", "achieved": round(achieved, 1), "peak": hbm,
            "unit": "GB/s", "frac": round(achieved / hbm, 4),
            "traffic": profiled_traffic(dname, inp.name),
            "peak_source": f"{peak_kind} hbm_gbs (MEASURED_PEAKS.json)",
            "alg_bytes_per_launch": dk["alg_bytes"]}

    parallelism = f"replicas x{nw}" if nw > 1 else "single device"
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": nw, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * el_max / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic", "config": workload_config(inp, {"parallelism": parallelism}),
            "l2": "inputs larger than L2: %.2f GB of expert weights streamed per step" % (
                (inp.E * 3 * inp.I * inp.H * 2) / 1e9),
            "plan": layer.plan,
            "e2e": {"value": e2e_tokens / e2e_max, "unit": UNIT, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h},
            "gpu_launches": args.steps * layer.plan["launches"],
            "clocks": clk, "roofline": roof, "kernels": kernels,
            "base_moe_ms_per_step": head.get("base_moe_ms_per_step"),
            "lora_marginal_us": head.get("lora_marginal_us")}
    line["stream_floor"] = stream_floor(stream)
    if args.layers > 1:
        line["multi_layer"] = multi_layer(m, inp, layer.W1, layer.W2, layer.lora, layer.lg,
                                          layer.ta, layer.x, layer.ws, args.layers,
                                          max(10, args.steps // 4), max(3, args.warmup // 4))
    if rank == 0 and nw == 1 and not args.no_cpu_baseline:
        rate, reps, el = cpu_oracle_rate(inp, args.cpu_seconds)
        line["cpu_baseline"] = {"value": rate, "unit": UNIT, "cores": cpu_cores(),
                                "kind": "oracle",
                                "sample": f"{reps} whole batches of {inp.T} tokens, "
                                          f"{el:.1f} s (fp64 NumPy oracle, weights pre-converted)",
                                **host_info()}
    # every other configuration of the pages' workloads: throughput and per-stage roofline
    # fractions (fewer steps; no CPU baseline)
    if rank == 0 and args.workloads != "none":
        from workloads import ALL_WORKLOAD_NAMES
        names = ALL_WORKLOAD_NAMES if args.workloads == "all" else args.workloads.split(",")
        wl = {inp.name: {k: v for k, v in head.items()}}
        del layer
        torch.cuda.empty_cache()
        for name in names:
            if name in wl:
                continue
            other = Layer(m, name, args.expand_mode)
            wl[name] = measure(other, args.extra_steps, 5, max(5, args.kernel_steps // 5),
                               stream, peaks)
            wl[name]["l2"] = ("fits in L2: launch-bound" if name == "tiny"
                              else "inputs larger than L2")
            del other
            torch.cuda.empty_cache()
        line["workloads"] = wl
    if rank == 0:
        print(json.dumps(line), flush=True)
    if nw > 1:
        dist.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--kernel-steps", type=int, default=50)
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--ref-budget-s", type=float, default=120.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--layers", type=int, default=4,
                    help="also chain this many layers (eager and one CUDA graph); < 2 skips it")
    ap.add_argument("--workloads", default="all",
                    help="'all', 'none' or a comma list: other workloads measured after the "
                         "headline one (fewer steps, no CPU baseline)")
    ap.add_argument("--extra-steps", type=int, default=20)
    ap.add_argument("--expand-mode", type=int, default=0, choices=[0, 1],
                    help="0: the chain the library picks; 1: the expand in kernels of its own")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
