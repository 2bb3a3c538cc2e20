"""Benchmark of the DyRA linear layer (one forward = one step) on synthetic inputs.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config c5] [--impl dyra|reference]
                    [--no-per-config] [--no-cpu-baseline]

Prints ONE JSON line (rank 0). The headline workload is c5, the largest configuration (LLM
prefill MLP up-projection, 4 x 2048 tokens, 4096 -> 12288, k 1024, r 256, Newton-Schulz);
"per_config" holds the same numbers for the ViT-B fc1 (c2), DINOv3 fc1 / fc2 (c3) and Monarch
(c4) layers. `value` is whole-job tokens/s = (tokens all ranks processed) / (max over ranks of
the mean device time of the K timed forwards). Every forward reads
its inputs from HBM: L2 is flushed (a write of 2x the L2 size) before each timed step,
outside the events that time it. Under torchrun each rank runs an independent replica of
the whole workload on its own GPU (the batch's samples are independent least-squares
problems, so there is no data-path collective): weak scaling.

`--impl reference` times the fp64 CPU oracle on the host cores on a bounded sample of the
same workload (rank 0 only) and prints the same line with "impl": "reference".
"""
from __future__ import annotations

import argparse
import dataclasses
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
# the workloads timed beside the headline one (each as its own entry of "per_config"); "c2_t2"
# is the ViT-B fc1 layer with two ALS iterations (summary page 3.3 / Figure 9)
PER_CONFIG = ["c2", "c3_fc1", "c3_fc2", "c4", "c6", "c2_t2"]


def bench_config(name):
    if name == "c2_t2":
        return dataclasses.replace(WL.get_config("c2"), name="c2_vitb16_fc1_als_t2", als_t=2.0)
    return WL.get_config(name)
_CSRC = "input_adaptive_rank_dyra_b300/csrc/"
# the source files that define each kernel of the forward (a recorded DRAM-traffic figure is
# used only while their hash matches the one recorded with it)
GEMM_SOURCES = [_CSRC + "tc_gemm.cu", _CSRC + "tc_gemm.cuh", _CSRC + "ptx.cuh"]
KERNEL_SOURCES = {"cg_solve": GEMM_SOURCES + [_CSRC + "sweep.cuh"],   # the inversion in its epilogue
                  "spd_invert": [_CSRC + "solve.cu", _CSRC + "kernels.cuh", _CSRC + "sweep.cuh"],
                  "spd_apply_c": [_CSRC + "solve.cu", _CSRC + "kernels.cuh"],
                  "ns_iterate": [_CSRC + "ns.cu", _CSRC + "ptx.cuh", _CSRC + "kernels.cuh"],
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
    if cfg.kind == "blast":     # k = blocks per side, t = middle rank: stage 1 X blockdiag(U)
        t = cfg.blast_t
        if name == "blast_stage1":
            return 2.0 * B * n * d * t, e * (B * n * d + d * t + B * n * k * t)
        if name == "xproj_L":
            return 2.0 * B * n * d * r, e * (B * n * d + d * r + B * n * r)
        if name == "fused_output":
            return (2.0 * B * n * (k * t + r) * m,
                    e * (B * n * (k * t + r) + k * t * m + B * r * m + B * n * m) + 4 * m)
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
    if name == "cg_solve":      # cg_c_gram with the inversion and C~ = G^-1 C in its epilogue
        return (2.0 * B * n * r * (d + r) + B * 2.0 * r ** 3 + B * 2.0 * r * r * d,
                e * (B * n * d + B * n * r) + 4 * (B * r * d + B * r * r)
                + (4 + e) * B * r * r + e * B * r * d)
    if name == "cg_c_gram":
        return 2.0 * B * n * r * (d + r), e * (B * n * d + B * n * r) + 4 * (B * r * d + B * r * r)
    if name == "spd_invert":    # r / 4 block sweeps: about r^3 FMA; G in, G^-1 out (fp32, bf16)
        return B * 2.0 * r ** 3, 4 * B * r * r + (4 + e) * B * r * r
    if name == "spd_apply_c":   # C~ = G^-1 C: G^-1 and C^T (fp32) in, C~ (bf16) out
        return B * 2.0 * r * r * d, 4 * (B * r * r + B * r * d) + e * B * r * d
    if name == "ginv_c":
        return 2.0 * B * r * r * d, 4 * (B * r * r + B * r * d) + e * B * r * d
    if name == "als_gram_r":    # H = R R^T
        return 2.0 * B * r * r * m, e * B * r * m + 4 * B * r * r
    if name == "als_q":         # Q = W_res R^T, fp32 out
        return 2.0 * B * d * m * r, e * (d * m + B * r * m) + 4 * B * d * r
    if name == "als_l_update":  # L = X P_s into T
        return 2.0 * B * n * d * r, e * (B * n * d + B * r * d + B * n * r)
    if name == "residual_product":
        return 2.0 * B * r * d * m, e * (B * r * d + d * m + B * r * m)
    if name == "fused_output":
        return 2.0 * B * n * (k + r) * m, e * (B * n * (k + r) + k * m + B * r * m + B * n * m) + 4 * m
    if name == "ns_iterate":    # the start from G, [E ; X] E per iteration (the last one
        #                         X E only), then G^-1 = D X D; the iterates stay in L2:
        #                         G in, G^-1 out (fp32 and bf16)
        t = cfg.ns_iters
        return (B * (4.0 * (t - 1) + 2.0) * r ** 3,
                4 * B * r * r + (4 + e) * B * r * r)
    return 0.0, 0.0


def layer_flops(cfg):
    """Algorithmic FLOPs of the whole one-step DyRA forward (per batch). Monarch: two
    block-diagonal factors of nb blocks (2 n d nb + 2 n m nb)."""
    B, n, d, m, k, r = cfg.batch, cfg.n, cfg.d, cfg.m, cfg.k, cfg.r
    static = 2.0 * n * (d * k + k * m)
    if cfg.kind == "blast":   # stage 1 block-diagonal; stages 2-3 as the coupled factor
        static = 2.0 * n * (d * cfg.blast_t + k * cfg.blast_t * m)
    r_update = 2.0 * n * r * r + 2.0 * n * r * d + 2.0 * r * d * m
    dyn = 2.0 * n * d * r + r_update + 2.0 * n * r * m
    for hs in range(2, int(round(2 * getattr(cfg, "als_t", 1.0)))):
        # L-update: R R^T, W_res R^T, apply of (R R^T)^-1, X P; R-update as above
        dyn += (2.0 * r * r * m + 2.0 * d * m * r + 2.0 * r * r * d + 2.0 * n * d * r
                if hs % 2 == 0 else r_update)
    return B * (static + dyn)


def layer_bytes(cfg):
    B, n, d, m, k, r = cfg.batch, cfg.n, cfg.d, cfg.m, cfg.k, cfg.r
    if cfg.kind == "monarch":
        weights = 2 * (d * k + k * m + d * r + d * m) + 4 * m
        acts = 2 * (B * n * d + B * n * m)
        inter = 2 * (3 * B * n * (d + r) + 2 * B * r * d + 2 * B * r * m) + 4 * B * r * r
        return weights + acts + inter
    if cfg.kind == "blast":
        k = k * cfg.blast_t
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
            ("cholesky" if cfg.r <= 64 else "newton_schulz"), "als_t": cfg.als_t,
            "l2": "flushed before every timed step (write of 2x L2)"}


# ---------------------------------------------------------------------------- CPU oracle

# Samples of each workload that one CPU pass of the oracle forward covers: enough tokens for a
# stable rate, few enough that a pass stays around a second on a many-core host.
ORACLE_SAMPLES = {"c1_fp32_single_layer": 1, "c2_vitb16_fc1": 4, "c3_dinov3_vitl16_fc1": 1,
                  "c3_dinov3_vitl16_fc2": 1, "c4_monarch32_attn_proj": 1, "c5_prefill_mlp_up": 1}


@functools.lru_cache(maxsize=None)
def _oracle_inputs(cfg):
    """Oracle preparation (untimed) and the first samples of the workload."""
    import oracle as O
    W, b = WL.make_weights(cfg)
    prep = O.prepare(W, b, cfg.kind, cfg.k, cfg.r)
    ns = min(cfg.batch, ORACLE_SAMPLES.get(cfg.name, 1))
    return prep, WL.make_inputs(cfg, range(ns))


def _cpu_model() -> str:
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def _openblas():
    """(get, set) thread-count functions of the OpenBLAS that numpy has loaded, found by its
    exported names, or None (used when threadpoolctl is not installed)."""
    import ctypes
    import re
    np.ones(2) @ np.ones(2)   # make sure the BLAS is loaded
    try:
        maps = open("/proc/self/maps").read()
    except OSError:
        return None
    for path in sorted(set(re.findall(r"(/\S*openblas\S*\.so\S*)", maps))):
        try:
            lib = ctypes.CDLL(path)
        except OSError:
            continue
        for pre in ("scipy_openblas", "openblas"):
            for suf in ("64_", "_64_", ""):
                g = getattr(lib, f"{pre}_get_num_threads{suf}", None)
                st = getattr(lib, f"{pre}_set_num_threads{suf}", None)
                if g is not None and st is not None:
                    g.restype = ctypes.c_int
                    st.argtypes = [ctypes.c_int]
                    return g, st
    return None


def _blas_threads() -> int:
    try:
        from threadpoolctl import threadpool_info
        return max([i.get("num_threads", 1) for i in threadpool_info()] or [1])
    except Exception:
        ob = _openblas()
        if ob is not None:
            return int(ob[0]())
        return os.cpu_count() or 1


class _one_blas_thread:
    """Limits numpy's BLAS to one thread inside the block (threadpoolctl, else OpenBLAS's own
    thread-count calls)."""

    def __enter__(self):
        self._ctx, self._ob, self._prev = None, None, None
        try:
            from threadpoolctl import threadpool_limits
            self._ctx = threadpool_limits(limits=1)
            self._ctx.__enter__()
            return self
        except ImportError:
            pass
        self._ob = _openblas()
        if self._ob is None:
            raise RuntimeError("no way to limit the BLAS thread count")
        self._prev = int(self._ob[0]())
        self._ob[1](1)
        return self

    def __exit__(self, *exc):
        if self._ctx is not None:
            self._ctx.__exit__(*exc)
        elif self._ob is not None:
            self._ob[1](self._prev)


def _solver_of(cfg) -> str:
    return cfg.solver if cfg.solver != "auto" else ("cholesky" if cfg.r <= 64 else "newton_schulz")


def oracle_pass(cfg):
    """One timed pass of the fp64 oracle's forward (fit excluded) over the bounded sample.
    Returns (tokens, seconds)."""
    import oracle as O
    prep, X = _oracle_inputs(cfg)
    t0 = time.perf_counter()
    O.forward(X, prep, solver=_solver_of(cfg), ns_iters=cfg.ns_iters)
    return X.shape[0] * cfg.n, time.perf_counter() - t0


def oracle_baseline(cfg, seconds: float = 10.0):
    """Times the fp64 oracle's forward on the bounded sample, repeated until `seconds` have
    passed, on all host threads; then one pass with the BLAS limited to one thread."""
    prep, X = _oracle_inputs(cfg)
    oracle_pass(cfg)   # warm-up
    tokens, el, reps = 0, 0.0, 0
    while el < seconds:
        t, dt = oracle_pass(cfg)
        tokens += t
        el += dt
        reps += 1
    one = None
    try:
        with _one_blas_thread():
            t1, dt1 = oracle_pass(cfg)
        one = {"value": t1 / dt1, "unit": "tokens/s", "cores": 1, "seconds": dt1}
    except Exception as e:   # reported, never fatal
        one = {"unavailable": f"{type(e).__name__}: {e}"}
    nsamp = X.shape[0]
    return {"value": tokens / el, "unit": "tokens/s", "cores": _blas_threads(), "kind": "oracle",
            "cpu_model": _cpu_model(), "host_cpus": os.cpu_count(),
            "sample": f"{nsamp} of {cfg.batch} samples ({nsamp * cfg.n} tokens) x {reps} passes, "
                      f"fp64 numpy/LAPACK forward, fit excluded, {el:.1f} s",
            "single_thread": one}


def run_reference(args, cfg):
    """The reference arm: the fp64 oracle on the host cores, one pass over the bounded sample
    per step (W untimed passes, then K timed ones); ms_per_step is the measured time of a
    step's pass and value its tokens per second (median over the steps)."""
    rank, world, _ = dist_init(args.gpus)
    if rank != 0:
        return
    for _ in range(args.warmup):
        oracle_pass(cfg)
    per_ms, per_rate = [], []
    tokens = 0
    for _ in range(args.steps):
        tokens, dt = oracle_pass(cfg)
        per_ms.append(dt * 1e3)
        per_rate.append(tokens / dt)
    value = statistics.median(per_rate)
    nsamp = tokens // cfg.n
    sample = (f"{nsamp} of {cfg.batch} samples ({tokens} tokens) per step, fp64 numpy/LAPACK "
              "forward, fit excluded")
    conf = dict(workload_config(cfg))
    conf["sample"] = sample
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": statistics.median(per_ms), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": conf,
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": _blas_threads(),
                             "kind": "oracle", "cpu_model": _cpu_model(), "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------- GPU arm

def _torch_input(cfg, X):
    import torch
    if cfg.dtype == "bf16":
        return torch.from_numpy(WL.bf16_bits(X).view(np.int16)).view(torch.bfloat16)
    return torch.from_numpy(X.astype(np.float32))


def measure_config(cfg, args, dev, world, pk, with_e2e: bool, clocks=None):
    """Times one configuration on this rank's GPU: the DyRA forward (CUDA-graph replays of
    one dyra_linear_forward call, L2 flushed before each step), its kernels one by one, the
    dense cuBLAS X W + b on the same input and, if asked, the host-buffer entry point."""
    import torch
    import input_adaptive_rank_dyra_b300 as dy
    W, b = WL.make_weights(cfg)
    t0 = time.perf_counter()
    layer = dy.prepare(W, b, kind=cfg.kind, k=cfg.k, r=cfg.r, dtype=cfg.dtype,
                       device=dev.index, solver=cfg.solver, ns_iters=cfg.ns_iters,
                       als_t=cfg.als_t, blast_t=cfg.blast_t)
    prep_s = time.perf_counter() - t0
    X = WL.make_inputs(cfg)
    tdt = torch.bfloat16 if cfg.dtype == "bf16" else torch.float32
    Xh = _torch_input(cfg, X)
    Xd = Xh.to(dev)
    Y = torch.empty((cfg.batch, cfg.n, cfg.m), dtype=tdt, device=dev)
    ws = dy.new_workspace(layer, cfg.batch, cfg.n)
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    nk = layer.kernels_per_forward
    names = layer.kernel_names()
    K, Wm = args.steps, args.warmup

    # Each timed step replays a CUDA graph captured from one dyra_linear_forward call, so the
    # GPU runs the step's kernels back to back with their programmatic-launch edges. A second
    # pass replays graphs of dyra_linear_forward_profiled, which put an event pair around
    # every kernel: the per-kernel times (the event nodes sit between kernels, so their sum
    # is not the step time).
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
    t0 = time.perf_counter()
    for _ in range(20):
        dy.linear_forward(layer, Xd, Y, ws)
    host_us = (time.perf_counter() - t0) / 20 * 1e6
    torch.cuda.synchronize()
    if clocks is not None:
        clocks.__enter__()
    t_start = time.perf_counter()
    i = 0
    # W warm-up replays at least, and enough of them (about a second) for the clock sampler
    # to see the GPU under load before the timed region
    while i < Wm or time.perf_counter() - t_start < args.clock_warmup_s:
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
    if clocks is not None:
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
        raise RuntimeError(f"{cfg.name}: {tmo} bounded waits timed out in the forward")
    ms_local = float(np.mean(step_ms))
    tokens = cfg.batch * cfg.n
    value, ms = weak_scaling_value(tokens, ms_local, world)

    # dense cuBLAS X W + b on the same input, same flushing
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
    del Wd, Yd

    out = {"cfg": cfg, "value": value, "ms": ms, "ms_local": ms_local, "dense_ms": dense_ms,
           "kern_ms": kern_ms, "names": names, "nk": nk, "host_us": host_us, "nsp": nsp,
           "prep_s": prep_s, "tokens": tokens}

    if with_e2e:
        # end to end through the host-buffer entry point (pinned host X and Y)
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
        out["e2e_ms"] = max_over_ranks(float(np.mean([est[i].elapsed_time(een[i])
                                                      for i in range(K)])), world)
    layer.close()
    del flush, Xd, Y, ws
    torch.cuda.empty_cache()
    return out


def measure_mlp(cfg1, cfg2, args, dev, world):
    """The DINOv3 MLP block, fc1 -> GELU -> fc2, with both layers replaced (one
    dyra_mlp_forward call, CUDA-graph replays, L2 flushed before each step), next to the dense
    block addmm -> gelu -> addmm (cuBLAS) on the same input."""
    import torch
    import input_adaptive_rank_dyra_b300 as dy
    W1, b1 = WL.make_weights(cfg1)
    W2, b2 = WL.make_weights(cfg2)
    fc1 = dy.prepare(W1, b1, kind=cfg1.kind, k=cfg1.k, r=cfg1.r, dtype="bf16", device=dev.index,
                     activation="gelu")
    fc2 = dy.prepare(W2, b2, kind=cfg2.kind, k=cfg2.k, r=cfg2.r, dtype="bf16", device=dev.index)
    X = WL.make_inputs(cfg1)
    Xd = _torch_input(cfg1, X).to(dev)
    B, n = cfg1.batch, cfg1.n
    H = torch.empty((B, n, cfg1.m), dtype=torch.bfloat16, device=dev)
    Y = torch.empty((B, n, cfg2.m), dtype=torch.bfloat16, device=dev)
    ws = torch.empty(max(fc1.workspace_size(B, n), fc2.workspace_size(B, n)), dtype=torch.uint8,
                     device=dev)
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    K, Wm = args.steps, args.warmup
    for _ in range(3):
        dy.mlp_forward(fc1, fc2, Xd, H, Y, ws)
    torch.cuda.synchronize()
    cap = torch.cuda.Stream(dev)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=cap):
        dy.mlp_forward(fc1, fc2, Xd, H, Y, ws, stream=cap)
    for _ in range(Wm):
        flush.fill_(1.0)
        g.replay()
    st = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    en = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    torch.cuda.synchronize()
    barrier(world)
    for i in range(K):
        flush.fill_(float(i))
        st[i].record(stream)
        g.replay()
        en[i].record(stream)
    torch.cuda.synchronize()
    ms = max_over_ranks(float(np.mean([st[i].elapsed_time(en[i]) for i in range(K)])), world)
    nsp, tmo = dy.workspace_status(fc2, ws)
    if tmo:
        raise RuntimeError(f"MLP block: {tmo} bounded waits timed out")
    W1d = torch.from_numpy(WL.bf16_bits(W1).view(np.int16)).view(torch.bfloat16).to(dev)
    W2d = torch.from_numpy(WL.bf16_bits(W2).view(np.int16)).view(torch.bfloat16).to(dev)
    b1d = torch.from_numpy(b1.astype(np.float32)).to(dev).to(torch.bfloat16)
    b2d = torch.from_numpy(b2.astype(np.float32)).to(dev).to(torch.bfloat16)
    X2 = Xd.view(-1, cfg1.d)
    Hd = torch.empty((B * n, cfg1.m), dtype=torch.bfloat16, device=dev)
    Yd = torch.empty((B * n, cfg2.m), dtype=torch.bfloat16, device=dev)

    def dense():
        torch.addmm(b1d, X2, W1d, out=Hd)
        Hg = torch.nn.functional.gelu(Hd)
        torch.addmm(b2d, Hg, W2d, out=Yd)

    for _ in range(Wm):
        flush.fill_(1.0)
        dense()
    for i in range(K):
        flush.fill_(float(i))
        st[i].record(stream)
        dense()
        en[i].record(stream)
    torch.cuda.synchronize()
    dense_ms = float(np.mean([st[i].elapsed_time(en[i]) for i in range(K)]))
    fl = layer_flops(cfg1) + layer_flops(cfg2)
    out = {"workload": "c3_dinov3_vitl16_mlp_block", "latency_us": ms * 1e3,
           "tokens_per_s": world * B * n / (ms * 1e-3),
           "tc_frac_of_peak": fl / (ms * 1e-3) / (peaks()[0]["bf16_tflops"] * 1e12),
           "dense_cublas": {"us": dense_ms * 1e3, "tokens_per_s": B * n / (dense_ms * 1e-3),
                            "speedup_of_dyra": dense_ms / ms,
                            "what": "addmm -> gelu -> addmm (bf16)"},
           "layers": [cfg1.name + " (GELU in its output epilogue)", cfg2.name],
           "not_spd_samples": nsp}
    fc1.close()
    fc2.close()
    return out


def summarize(res, pk, pk_kind):
    """The per-configuration numbers: latency, dense reference, TC and roofline fractions,
    per-kernel times (keyed by launch index) and the roofline of the dominant kernel."""
    cfg = res["cfg"]
    names, kern_ms, nk = res["names"], res["kern_ms"], res["nk"]
    ms = res["ms"]
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
    roof["launch_index"] = top
    roof["kernel_us"] = mean_k[top] * 1e3
    roof["algorithmic_bytes"] = by
    roof["algorithmic_flops"] = fl
    roof["peak_source"] = (f"{pk_kind} (MEASURED_PEAKS.json burst: the kernel runs well under "
                           "a millisecond)") if pk_kind == "measured" else "fallback"
    fl_layer = layer_flops(cfg)
    t_layer = ms * 1e-3
    t_roof = max(fl_layer / (tc_peak * 1e12), layer_bytes(cfg) / (hbm_peak * 1e9))
    kernels = []
    for j in range(nk):
        f, b_ = kernel_work(cfg, names[j])
        t = float(mean_k[j]) * 1e-3
        kernels.append({"i": j, "name": names[j], "us": round(float(mean_k[j]) * 1e3, 3),
                        "tflops": round(f / t / 1e12, 1) if f else 0.0,
                        "gbs": round(b_ / t / 1e9, 1) if b_ else 0.0})
    return {
        "workload": cfg.name, "latency_us": ms * 1e3, "tokens_per_s": res["value"],
        "tc_frac_of_peak": fl_layer / t_layer / (tc_peak * 1e12),
        "layer_roofline_frac": t_roof / t_layer,
        "layer_tflops": fl_layer / t_layer / 1e12,
        "dense_cublas": {"us": res["dense_ms"] * 1e3,
                         "tokens_per_s": res["tokens"] / (res["dense_ms"] * 1e-3),
                         "speedup_of_dyra": res["dense_ms"] / res["ms_local"]},
        "kernels_us": kernels, "roofline": roof,
        "not_spd_samples": res["nsp"], "prepare_s": res["prep_s"],
    }


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

    clocks = ClockSampler(local)
    head = measure_config(cfg, args, dev, world, pk, with_e2e=True, clocks=clocks)
    h = summarize(head, pk, pk_kind)
    others = []
    if not args.no_per_config:
        for name in PER_CONFIG:
            c = bench_config(name)
            if c.name == cfg.name:
                continue
            others.append(summarize(measure_config(c, args, dev, world, pk, with_e2e=False),
                                    pk, pk_kind))
        others.append(measure_mlp(WL.get_config("c3_fc1"), WL.get_config("c3_fc2"), args, dev,
                                  world))
    tokens = head["tokens"]
    ebytes = 2 if cfg.dtype == "bf16" else 4
    line = {
        "metric": METRIC, "value": head["value"], "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": head["ms"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": cfg.dtype,
        "data": "synthetic (seeded; no dataset)", "config": workload_config(cfg),
        "latency_us": h["latency_us"], "tc_frac_of_peak": h["tc_frac_of_peak"],
        "layer_roofline_frac": h["layer_roofline_frac"], "layer_tflops": h["layer_tflops"],
        "dense_cublas": h["dense_cublas"], "kernels_us": h["kernels_us"],
        "roofline": h["roofline"],
        "e2e": {"value": world * tokens / (head["e2e_ms"] * 1e-3), "unit": "tokens/s",
                "h2d_bytes_per_step": tokens * cfg.d * ebytes,
                "d2h_bytes_per_step": tokens * cfg.m * ebytes},
        "gpu_launches": args.steps * head["nk"],
        "host_enqueue_us": head["host_us"],
        "clocks": clocks.summary(),
        "not_spd_samples": head["nsp"],
        "prepare_s": head["prep_s"],
        "per_config": others,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = oracle_baseline(cfg)
    if rank == 0:
        print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--config", default="c5", choices=sorted(WL.CONFIGS),
                    help="headline workload (default: c5, the largest)")
    ap.add_argument("--impl", default="dyra", choices=["dyra", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true",
                    help="time only the headline workload")
    ap.add_argument("--clock-warmup-s", type=float, default=1.0,
                    help="seconds of warm-up replays before the timed region (0: only W of "
                         "them, e.g. under a profiler)")
    ap.add_argument("--batch", type=int, default=None,
                    help="samples per step instead of the workload's own (smaller profiler "
                         "captures; the line's config then names the reduced batch)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    cfg = WL.get_config(args.config)
    if args.batch is not None:
        if args.batch < 1:
            ap.error("--batch must be >= 1")
        cfg = dataclasses.replace(cfg, batch=args.batch, name=f"{cfg.name}_batch{args.batch}")
    if args.impl == "reference":
        run_reference(args, cfg)
    else:
        run_dyra(args, cfg)


if __name__ == "__main__":
    main()
