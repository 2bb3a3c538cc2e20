"""Benchmark of the DyRA linear layer (one forward = one step) on synthetic inputs.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config c2] [--impl dyra|reference]

Prints ONE JSON line (rank 0). `value` is whole-job tokens/s = (tokens all ranks processed)
/ (max over ranks of the summed device time of the K timed forwards). Every forward reads
its inputs from HBM: L2 is flushed (a write of 2x the L2 size) before each timed step,
outside the events that time it. Under torchrun each rank runs an independent replica of
the whole workload on its own GPU (the batch's samples are independent least-squares
problems, so there is no data-path collective): weak scaling.

`--impl reference` times the fp64 CPU oracle on the host cores on a bounded sample of the
same workload (rank 0 only) and prints the same line with "impl": "reference".
"""
from __future__ import annotations

import argparse
import functools
import hashlib
import json
import os
import statistics
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads as WL  # noqa: E402

METRIC = "DyRA layer tokens/s and latency vs dense cuBLAS XW; % bf16 TC peak"
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}
L2_BYTES = 126 * 1024 * 1024
_CSRC = "input_adaptive_rank_dyra_b300/csrc/"
# the source files that define each kernel of the forward (a recorded DRAM-traffic figure is
# used only while their hash matches the one recorded with it)
GEMM_SOURCES = [_CSRC + "tc_gemm.cu", _CSRC + "tc_gemm.cuh", _CSRC + "ptx.cuh"]
KERNEL_SOURCES = {"spd_solve_c": [_CSRC + "solve.cu", _CSRC + "kernels.cuh"],
                  "ns_prep": [_CSRC + "solve.cu"], "ns_finish": [_CSRC + "solve.cu"],
                  "monarch_permute": [_CSRC + "monarch.cu", _CSRC + "monarch.cuh"]}


# ---------------------------------------------------------------------------- helpers

def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def kernel_source_hash(kernel: str) -> str:
    """Hash of the kernel's source files with // comments and blank space removed, so that
    editing a comment does not invalidate a recorded capture."""
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES.get(kernel, GEMM_SOURCES):
        with open(os.path.join(ROOT, rel), encoding="utf-8") as f:
            for line in f:
                code = line.split("//", 1)[0].strip()
                if code:
                    h.update(code.encode() + b"\n")
    return h.hexdigest()[:12]


def recorded_traffic(workload: str, kernel: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on the current
    kernel sources (else None)."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(p):
        return None
    cur = kernel_source_hash(kernel)
    with open(p) as f:
        for line in f:
            parts = line.split()
            if len(parts) >= 4 and not line.startswith("#"):
                if parts[0] == workload and parts[1] == kernel and parts[3] == cur:
                    return float(parts[2])
    return None


def kernel_work(cfg, name: str):
    """Algorithmic (FLOPs, bytes) of one launch of kernel `name` over the whole batch.
    Bytes count each operand read once and each result written once, in its storage type
    (bf16 = 2 B; G fp32)."""
    B, n, d, m, k, r = cfg.batch, cfg.n, cfg.d, cfg.m, cfg.k, cfg.r
    e = 2
    if cfg.kind == "monarch":   # k = number of blocks; Z = X BD1 has nb * nb = d columns
        if name == "monarch_bd1":
            return 2.0 * B * n * d * k, e * (2 * B * n * d + d * k)
        if name == "xproj_L":
            return 2.0 * B * n * d * r, e * (B * n * d + d * r + B * n * r)
        if name == "monarch_permute":
            return 0.0, e * 2 * B * n * d
        if name == "fused_output":
            return (2.0 * B * n * m * (k + r),
                    e * (B * n * (d + r) + m * k + B * r * m + B * n * m) + 4 * m)
    if name == "xproj_static_L":
        return 2.0 * B * n * d * (k + r), e * (B * n * d + (k + r) * d + B * n * (k + r))
    if name == "cg_c_gram":
        return 2.0 * B * n * r * (d + r), e * (B * n * d + B * n * r) + 4 * (B * r * d + B * r * r)
    if name == "spd_solve_c":   # r sweeps (r^3 FMA) + G^-1 applied to d columns
        return (B * (2.0 * r ** 3 + 2.0 * r * r * d),
                4 * (B * r * r + B * r * d) + e * (B * r * d + B * r * r))
    if name == "ginv_c":
        return 2.0 * B * r * r * d, 4 * (B * r * r + B * r * d) + e * B * r * d
    if name == "residual_product":
        return 2.0 * B * r * d * m, e * (B * r * d + d * m + B * r * m)
    if name == "fused_output":
        return 2.0 * B * n * (k + r) * m, e * (B * n * (k + r) + k * m + B * r * m + B * n * m) + 4 * m
    if name.startswith("ns_"):
        return 2.0 * B * r * r * r, 4 * 3 * B * r * r
    return 0.0, 0.0


def layer_flops(cfg):
    """Algorithmic FLOPs of the whole one-step DyRA forward (per batch). Monarch: two
    block-diagonal factors of nb blocks (2 n d nb + 2 n m nb)."""
    B, n, d, m, k, r = cfg.batch, cfg.n, cfg.d, cfg.m, cfg.k, cfg.r
    static = 2.0 * n * (d * k + k * m)
    dyn = 2.0 * n * d * r + 2.0 * n * r * r + 2.0 * n * r * d + 2.0 * r * d * m + 2.0 * n * r * m
    return B * (static + dyn)


def layer_bytes(cfg):
    B, n, d, m, k, r = cfg.batch, cfg.n, cfg.d, cfg.m, cfg.k, cfg.r
    if cfg.kind == "monarch":
        weights = 2 * (d * k + k * m + d * r + d * m) + 4 * m
        acts = 2 * (B * n * d + B * n * m)
        inter = 2 * (3 * B * n * (d + r) + 2 * B * r * d + 2 * B * r * m) + 4 * B * r * r
        return weights + acts + inter
    weights = 2 * (d * (k + r) + k * m + d * m) + 4 * m
    acts = 2 * (B * n * d + B * n * m)
    inter = 2 * (2 * B * n * (k + r) + 2 * B * r * d + 2 * B * r * m) + 4 * B * r * r
    return weights + acts + inter


class ClockSampler:
    """Samples the SM clock and the clock-event reasons while the timed region runs: through
    NVML when pynvml is importable, else from an `nvidia-smi -lms` subprocess."""
    REASONS = {"gpu_idle": 0x1, "applications_clocks_setting": 0x2, "sw_power_cap": 0x4,
               "hw_slowdown": 0x8, "sync_boost": 0x10, "sw_thermal_slowdown": 0x20,
               "hw_thermal_slowdown": 0x40, "hw_power_brake_slowdown": 0x80}

    def __init__(self, device_index: int, period_s: float = 0.002):
        self.samples, self.reasons, self.ok = [], set(), False
        self.max_mhz = None
        self.error = None
        self.source = None
        self._stop = threading.Event()
        self._period = period_s
        self._t = None
        self._proc = None
        self._bus = None
        try:
            import torch
            pr = torch.cuda.get_device_properties(device_index)
            self._bus = f"{pr.pci_domain_id:08x}:{pr.pci_bus_id:02x}:{pr.pci_device_id:02x}.0"
        except Exception as e:
            self.error = f"{type(e).__name__}: {e}"
        try:
            import pynvml
            pynvml.nvmlInit()
            self._nv = pynvml
            try:
                self._h = pynvml.nvmlDeviceGetHandleByPciBusId(self._bus.encode())
            except Exception:
                self._h = pynvml.nvmlDeviceGetHandleByIndex(device_index)
            self.max_mhz = pynvml.nvmlDeviceGetMaxClockInfo(self._h, pynvml.NVML_CLOCK_SM)
            self.ok, self.source = True, "nvml"
        except Exception as e:   # reported in the JSON line, never fatal
            self.error = f"{type(e).__name__}: {e}"
            if self._bus is not None:
                self.ok, self.source = True, "nvidia-smi"

    def _run(self):
        nv = self._nv
        get = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            nv.nvmlDeviceGetCurrentClocksThrottleReasons
        while not self._stop.is_set():
            try:
                self.samples.append(nv.nvmlDeviceGetClockInfo(self._h, nv.NVML_CLOCK_SM))
                self._add_mask(get(self._h))
            except Exception:
                pass
            time.sleep(self._period)

    def _add_mask(self, mask: int):
        for name, bit in self.REASONS.items():
            if mask & bit and name != "gpu_idle":
                self.reasons.add(name)

    def __enter__(self):
        if not self.ok:
            return self
        if self.source == "nvml":
            self._t = threading.Thread(target=self._run, daemon=True)
            self._t.start()
        else:
            import subprocess
            cmd = ["nvidia-smi", "-i", self._bus,
                   "--query-gpu=clocks.sm,clocks.max.sm,clocks_event_reasons.active",
                   "--format=csv,noheader,nounits", "-lms", "50"]
            try:
                self._proc = subprocess.Popen(cmd, stdout=subprocess.PIPE,
                                              stderr=subprocess.DEVNULL, text=True)
            except Exception as e:
                self.ok, self.error = False, f"{type(e).__name__}: {e}"
        return self

    def __exit__(self, *exc):
        if self._t is not None:
            self._stop.set()
            self._t.join()
        if self._proc is not None:
            self._proc.terminate()
            try:
                out, _ = self._proc.communicate(timeout=5)
            except Exception:
                self._proc.kill()
                out, _ = self._proc.communicate()
            for line in out.splitlines():
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 3:
                    continue
                try:
                    self.samples.append(float(parts[0]))
                    self.max_mhz = float(parts[1])
                    self._add_mask(int(parts[2], 16))
                except ValueError:
                    continue

    def summary(self):
        if not self.ok:
            return {"sm_mhz": None, "sm_max_mhz": None,
                    "reasons": [f"clock sampling unavailable: {self.error}"]}
        med = statistics.median(self.samples) if self.samples else None
        return {"sm_mhz": med, "sm_max_mhz": self.max_mhz, "reasons": sorted(self.reasons),
                "samples": len(self.samples), "source": self.source}


def dist_init(gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl"
        try:
            import torch
            if not torch.cuda.is_available():
                backend = "gloo"
        except Exception:
            backend = "gloo"
        dist.init_process_group(backend=backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def weak_scaling_value(tokens_per_rank: int, ms_local: float, world: int):
    """Whole-job throughput of `world` independent replicas: every rank processed
    tokens_per_rank tokens per step; the step time is the slowest rank's. Returns
    (tokens/s, the max-over-ranks ms)."""
    ms = max_over_ranks(ms_local, world)
    return world * tokens_per_rank / (ms * 1e-3), ms


def workload_config(cfg):
    return {"workload": cfg.name, "batch": cfg.batch, "n_tokens": cfg.n, "d": cfg.d, "m": cfg.m,
            "static": cfg.kind, "k": cfg.k, "r": cfg.r,
            "solver": cfg.solver if cfg.solver != "auto" else
            ("cholesky" if cfg.r <= 64 else "newton_schulz"),
            "l2": "flushed before every timed step (write of 2x L2)"}


# ---------------------------------------------------------------------------- CPU oracle

@functools.lru_cache(maxsize=None)
def _oracle_inputs(cfg):
    """Oracle preparation (untimed) and the first few samples of the workload."""
    import oracle as O
    W, b = WL.make_weights(cfg)
    prep = O.prepare(W, b, cfg.kind, cfg.k, cfg.r)
    return prep, WL.make_inputs(cfg, range(min(cfg.batch, 4)))


def oracle_baseline(cfg, seconds: float = 12.0):
    """Times the fp64 oracle's forward (the offline fit excluded) on a bounded sample of the
    workload: whole samples, repeated until `seconds` of CPU time have passed."""
    import oracle as O
    try:
        from threadpoolctl import threadpool_info
        cores = max([i.get("num_threads", 1) for i in threadpool_info()] or [1])
    except Exception:
        cores = os.cpu_count()
    prep, X = _oracle_inputs(cfg)
    solver = cfg.solver if cfg.solver != "auto" else ("cholesky" if cfg.r <= 64 else "newton_schulz")
    nsamp = X.shape[0]
    O.forward(X[:1], prep, solver=solver, ns_iters=cfg.ns_iters)   # warm-up
    t0 = time.perf_counter()
    tokens = 0
    reps = 0
    while True:
        O.forward(X, prep, solver=solver, ns_iters=cfg.ns_iters)
        tokens += nsamp * cfg.n
        reps += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    return {"value": tokens / el, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"{nsamp} of {cfg.batch} samples ({nsamp * cfg.n} tokens) x {reps} passes, "
                      f"fp64 numpy/LAPACK forward, fit excluded, {el:.1f} s"}


def run_reference(args, cfg):
    rank, world, _ = dist_init(args.gpus)
    if rank != 0:
        return
    per_step = []
    cb = None
    for _ in range(args.warmup):
        oracle_baseline(cfg, seconds=0.0)
    for _ in range(args.steps):
        cb = oracle_baseline(cfg, seconds=max(1.0, 20.0 / max(args.steps, 1)))
        per_step.append(cb["value"])
    value = statistics.median(per_step)
    cb["value"] = value
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": cfg.batch * cfg.n / value * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(cfg), "cpu_baseline": cb,
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------- GPU arm

def run_dyra(args, cfg):
    import torch
    import input_adaptive_rank_dyra_b300 as dy
    rank, world, local = dist_init(args.gpus)
    if not torch.cuda.is_available():
        raise RuntimeError("bench.py needs a CUDA device (B300)")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dy.load()
    pk, pk_kind = peaks()

    W, b = WL.make_weights(cfg)
    t0 = time.perf_counter()
    layer = dy.prepare(W, b, kind=cfg.kind, k=cfg.k, r=cfg.r, dtype=cfg.dtype, device=local,
                       solver=cfg.solver, ns_iters=cfg.ns_iters)
    prep_s = time.perf_counter() - t0
    X = WL.make_inputs(cfg)
    tdt = torch.bfloat16 if cfg.dtype == "bf16" else torch.float32
    if cfg.dtype == "bf16":
        Xh = torch.from_numpy(WL.bf16_bits(X).view(np.int16)).view(torch.bfloat16)
    else:
        Xh = torch.from_numpy(X.astype(np.float32))
    Xd = Xh.to(dev)
    Y = torch.empty((cfg.batch, cfg.n, cfg.m), dtype=tdt, device=dev)
    ws = dy.new_workspace(layer, cfg.batch, cfg.n)
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    nk = layer.kernels_per_forward
    names = layer.kernel_names()
    K, Wm = args.steps, args.warmup

    # ---- device-resident timed region. Each timed step replays a CUDA graph of one forward
    # captured from the same C-ABI call (dyra_linear_forward), so the GPU runs the step's
    # kernels back to back, with their programmatic-launch edges, instead of waiting on host
    # launches. A second pass replays graphs of dyra_linear_forward_profiled, which carry a
    # start/end event pair around every kernel on the stream that kernel runs on: it gives
    # the per-kernel times (the event nodes sit between kernels, so it is not the step time).
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2 * nk)] for _ in range(K)]
    st = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    en = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    for _ in range(3):   # builds and caches the launch plan before capture
        dy.linear_forward(layer, Xd, Y, ws)
        dy.linear_forward_profiled(layer, Xd, Y, ws, ev[0])
    torch.cuda.synchronize()
    cap = torch.cuda.Stream(dev)
    g_plain = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_plain, stream=cap):
        dy.linear_forward(layer, Xd, Y, ws, stream=cap)
    graphs = []
    for i in range(K):
        g = torch.cuda.CUDAGraph()
        for e in ev[i]:
            e.record(cap)
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=cap):
            dy.linear_forward_profiled(layer, Xd, Y, ws, ev[i], stream=cap)
        graphs.append(g)
    torch.cuda.synchronize()
    # host cost of one forward call (enqueue only), for reference
    t0 = time.perf_counter()
    for _ in range(20):
        dy.linear_forward(layer, Xd, Y, ws)
    host_us = (time.perf_counter() - t0) / 20 * 1e6
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    clocks.__enter__()
    t_start = time.perf_counter()
    i = 0
    # W warm-up replays at least, and enough of them (about a second) for the clock sampler
    # to see the GPU under load before the timed region
    while i < Wm or time.perf_counter() - t_start < 1.0:
        flush.fill_(1.0)
        g_plain.replay()
        i += 1
        if i % 50 == 0:
            torch.cuda.synchronize()
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    for i in range(K):
        flush.fill_(float(i))
        st[i].record(stream)
        g_plain.replay()
        en[i].record(stream)
    torch.cuda.synchronize()
    clocks.__exit__(None, None, None)
    barrier(world)
    torch.cuda.synchronize()
    step_ms = [st[i].elapsed_time(en[i]) for i in range(K)]
    for i in range(K):
        flush.fill_(float(i))
        graphs[i].replay()
    torch.cuda.synchronize()
    kern_ms = np.array([[ev[i][2 * j].elapsed_time(ev[i][2 * j + 1]) for j in range(nk)]
                        for i in range(K)])
    nsp, tmo = dy.workspace_status(layer, ws)
    if tmo:
        raise RuntimeError(f"{tmo} bounded waits timed out in the forward")
    ms_local = float(np.mean(step_ms))
    tokens = cfg.batch * cfg.n
    value, ms = weak_scaling_value(tokens, ms_local, world)

    # ---- dense cuBLAS XW + b on the same input, same flushing
    Wd = torch.from_numpy(WL.bf16_bits(W).view(np.int16)).view(torch.bfloat16).to(dev) \
        if cfg.dtype == "bf16" else torch.from_numpy(W.astype(np.float32)).to(dev)
    bd = torch.from_numpy(b.astype(np.float32)).to(dev).to(tdt)
    X2 = Xd.view(-1, cfg.d)
    Yd = torch.empty((tokens, cfg.m), dtype=tdt, device=dev)
    for _ in range(Wm):
        flush.fill_(1.0)
        torch.addmm(bd, X2, Wd, out=Yd)
    dst = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    den = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    for i in range(K):
        flush.fill_(float(i))
        dst[i].record(stream)
        torch.addmm(bd, X2, Wd, out=Yd)
        den[i].record(stream)
    torch.cuda.synchronize()
    dense_ms = float(np.mean([dst[i].elapsed_time(den[i]) for i in range(K)]))

    # ---- end to end through the host-buffer entry point (pinned host X and Y)
    Xp = Xh.pin_memory()
    Yp = torch.empty((cfg.batch, cfg.n, cfg.m), dtype=tdt).pin_memory()
    Xs = torch.empty_like(Xd)
    for _ in range(Wm):
        dy.linear_forward_host(layer, Xp, Yp, Xs, Y, ws)
    torch.cuda.synchronize()
    est = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    een = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    for i in range(K):
        flush.fill_(float(i))
        est[i].record(stream)
        dy.linear_forward_host(layer, Xp, Yp, Xs, Y, ws)
        een[i].record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(float(np.mean([est[i].elapsed_time(een[i]) for i in range(K)])), world)
    ebytes = 2 if cfg.dtype == "bf16" else 4

    # ---- roofline of the dominant kernel
    mean_k = kern_ms.mean(axis=0)
    top = int(np.argmax(mean_k))
    top_name = names[top]
    fl, by = kernel_work(cfg, top_name)
    t_s = mean_k[top] * 1e-3
    tc_peak, hbm_peak = pk["bf16_tflops"], pk["hbm_gbs"]
    if by / (hbm_peak * 1e9) >= fl / (tc_peak * 1e12):
        roof = {"bound": "hbm", "achieved": by / t_s / 1e9, "peak": hbm_peak, "unit": "GB/s"}
    else:
        roof = {"bound": "tensor", "achieved": fl / t_s / 1e12, "peak": tc_peak, "unit": "TFLOP/s"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["traffic"] = recorded_traffic(cfg.name, top_name)
    roof["kernel"] = top_name
    roof["kernel_us"] = mean_k[top] * 1e3
    roof["algorithmic_bytes"] = by
    roof["algorithmic_flops"] = fl
    roof["peak_source"] = f"{pk_kind} (MEASURED_PEAKS.json burst)" if pk_kind == "measured" \
        else "fallback"

    fl_layer = layer_flops(cfg)
    t_layer = ms * 1e-3
    t_roof = max(fl_layer / (tc_peak * 1e12), layer_bytes(cfg) / (hbm_peak * 1e9))
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": K,
        "warmup": Wm, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": cfg.dtype, "data": "synthetic (seeded; no dataset)",
        "config": workload_config(cfg),
        "latency_us": ms * 1e3,
        "tc_frac_of_peak": fl_layer / t_layer / (tc_peak * 1e12),
        "layer_roofline_frac": t_roof / t_layer,
        "layer_tflops": fl_layer / t_layer / 1e12,
        "dense_cublas": {"us": dense_ms * 1e3, "tokens_per_s": tokens / (dense_ms * 1e-3),
                         "speedup_of_dyra": dense_ms / ms_local},
        "kernels_us": {names[j]: round(float(mean_k[j]) * 1e3, 3) for j in range(nk)},
        "roofline": roof,
        "e2e": {"value": world * tokens / (e2e_ms * 1e-3), "unit": "tokens/s",
                "h2d_bytes_per_step": tokens * cfg.d * ebytes,
                "d2h_bytes_per_step": tokens * cfg.m * ebytes},
        "gpu_launches": K * nk,
        "host_enqueue_us": host_us,
        "clocks": clocks.summary(),
        "not_spd_samples": nsp,
        "prepare_s": prep_s,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = oracle_baseline(cfg)
    if rank == 0:
        print(json.dumps(line), flush=True)
    layer.close()


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--config", default="c2", choices=sorted(WL.CONFIGS))
    ap.add_argument("--impl", default="dyra", choices=["dyra", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    cfg = WL.get_config(args.config)
    if args.impl == "reference":
        run_reference(args, cfg)
    else:
        run_dyra(args, cfg)


if __name__ == "__main__":
    main()
