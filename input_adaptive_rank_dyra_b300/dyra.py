"""Python binding of the DyRA C ABI (include/dyra.h), by ctypes.

Argument marshalling only: every step of the layer runs in the CUDA kernels of
``libdyra_b300.so``. PyTorch supplies device memory and streams. If the shared library
is missing or cannot be loaded, every call raises; there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libdyra_b300.so")

DYRA_OK = 0
STATUS_NAMES = {0: "OK", 1: "INVALID_ARG", 2: "UNSUPPORTED", 3: "CUDA", 4: "OOM", 5: "NOT_SPD",
                6: "TIMEOUT", 7: "WORKSPACE", 8: "NO_DEVICE"}
KINDS = {"lowrank": 0, "monarch": 1, "blast": 2}
DTYPES = {"f32": 0, "bf16": 1}
SOLVERS = {"auto": 0, "cholesky": 1, "newton_schulz": 2}
INPUT_AWARE = {None: 0, "none": 0, "diag": 1, "cholesky": 2}
ACTIVATIONS = {None: 0, "none": 0, "gelu": 1}
BUFFERS = {"T": 0, "C": 1, "G": 2, "GINV": 3, "B": 4, "R": 5, "CS": 6}

_c_double_p = ctypes.POINTER(ctypes.c_double)


class PrepareArgs(ctypes.Structure):
    _fields_ = [
        ("W", _c_double_p), ("b", _c_double_p), ("d", ctypes.c_int), ("m", ctypes.c_int),
        ("kind", ctypes.c_int), ("k", ctypes.c_int), ("r", ctypes.c_int), ("R0", _c_double_p),
        ("F1", _c_double_p), ("F2", _c_double_p), ("ridge", ctypes.c_double),
        ("solver", ctypes.c_int), ("ns_iters", ctypes.c_int), ("dtype", ctypes.c_int),
        ("device", ctypes.c_int), ("fit_threads", ctypes.c_int), ("calib", _c_double_p),
        ("n_calib", ctypes.c_int), ("input_aware", ctypes.c_int), ("activation", ctypes.c_int),
        ("als_t", ctypes.c_double), ("blast_t", ctypes.c_int), ("F3", _c_double_p),
    ]


class LayerDesc(ctypes.Structure):
    _fields_ = [
        ("d", ctypes.c_int), ("m", ctypes.c_int), ("k", ctypes.c_int), ("r", ctypes.c_int),
        ("kind", ctypes.c_int), ("dtype", ctypes.c_int), ("solver", ctypes.c_int),
        ("ns_iters", ctypes.c_int), ("ridge", ctypes.c_double), ("device", ctypes.c_int),
        ("kernels_per_forward", ctypes.c_int), ("activation", ctypes.c_int),
        ("als_t", ctypes.c_double),
    ]


EXPORTED = [
    "dyra_prepare", "dyra_fit", "dyra_layer_destroy", "dyra_layer_info", "dyra_export",
    "dyra_export_factors", "dyra_workspace_size", "dyra_linear_forward",
    "dyra_linear_forward_host", "dyra_linear_forward_profiled", "dyra_kernel_name",
    "dyra_workspace_status", "dyra_workspace_tensor", "dyra_status_string", "dyra_last_error",
    "dyra_abi_version", "dyra_linear_forward_static", "dyra_selftest_bounded_wait",
    "dyra_mlp_forward",
]

_lib = None


class DyraError(RuntimeError):
    def __init__(self, status: int, where: str):
        msg = f"{where}: {STATUS_NAMES.get(status, status)}"
        if _lib is not None:
            detail = _lib.dyra_last_error().decode()
            if detail:
                msg += f" ({detail})"
        super().__init__(msg)
        self.status = status


def load(path: Optional[str] = None) -> ctypes.CDLL:
    """Load the shared library (once). Raises if it is missing."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"{p} is missing: build it with "
                           "`python -m input_adaptive_rank_dyra_b300.build`")
    lib = ctypes.CDLL(p)
    vp, i, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    lib.dyra_prepare.argtypes = [ctypes.POINTER(PrepareArgs), ctypes.POINTER(vp)]
    lib.dyra_fit.argtypes = [ctypes.POINTER(PrepareArgs), vp, vp, vp, vp, vp, vp]
    lib.dyra_layer_destroy.argtypes = [vp]
    lib.dyra_layer_destroy.restype = None
    lib.dyra_layer_info.argtypes = [vp, ctypes.POINTER(LayerDesc)]
    lib.dyra_export.argtypes = [vp, vp, vp, vp, vp]
    lib.dyra_export_factors.argtypes = [vp, vp, vp]
    lib.dyra_workspace_size.argtypes = [vp, i, i, ctypes.POINTER(sz)]
    lib.dyra_linear_forward.argtypes = [vp, vp, i, i, vp, vp, sz, vp]
    lib.dyra_linear_forward_host.argtypes = [vp, vp, i, i, vp, vp, vp, vp, sz, vp]
    lib.dyra_linear_forward_profiled.argtypes = [vp, vp, i, i, vp, vp, sz, vp,
                                                 ctypes.POINTER(vp), i, ctypes.POINTER(i)]
    lib.dyra_kernel_name.argtypes = [vp, i]
    lib.dyra_kernel_name.restype = ctypes.c_char_p
    lib.dyra_workspace_status.argtypes = [vp, vp, vp, ctypes.POINTER(i), ctypes.POINTER(i)]
    lib.dyra_workspace_tensor.argtypes = [vp, i, i, i, ctypes.POINTER(sz), ctypes.POINTER(i)]
    lib.dyra_status_string.argtypes = [i]
    lib.dyra_status_string.restype = ctypes.c_char_p
    lib.dyra_last_error.argtypes = []
    lib.dyra_last_error.restype = ctypes.c_char_p
    lib.dyra_abi_version.argtypes = []
    lib.dyra_linear_forward_static.argtypes = [vp, vp, i, i, vp, vp]
    lib.dyra_selftest_bounded_wait.argtypes = [i, vp, vp]
    lib.dyra_mlp_forward.argtypes = [vp, vp, vp, i, i, vp, vp, vp, sz, vp]
    for name in EXPORTED:   # raises AttributeError if the library lacks an entry point
        getattr(lib, name)
    if path is None:
        _lib = lib
    return lib


def _check(status: int, where: str):
    if status != DYRA_OK:
        raise DyraError(status, where)


def _f64(a, shape=None):
    if a is None:
        return None
    arr = np.ascontiguousarray(np.asarray(a, dtype=np.float64))
    if shape is not None and arr.shape != tuple(shape):
        raise ValueError(f"expected shape {shape}, got {arr.shape}")
    return arr


def _ptr(arr):
    return None if arr is None else arr.ctypes.data_as(_c_double_p)


def _stream_handle(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


class Layer:
    """A prepared DyRA layer (owns the C handle)."""

    def __init__(self, handle: ctypes.c_void_p):
        self._h = handle
        d = LayerDesc()
        _check(load().dyra_layer_info(self._h, ctypes.byref(d)), "dyra_layer_info")
        self.desc = d
        self.d, self.m, self.k, self.r = d.d, d.m, d.k, d.r
        self.kind = {v: k for k, v in KINDS.items()}[d.kind]
        self.dtype = {v: k for k, v in DTYPES.items()}[d.dtype]
        self.solver = {v: k for k, v in SOLVERS.items()}[d.solver]
        self.ns_iters = d.ns_iters
        self.device = d.device
        self.kernels_per_forward = d.kernels_per_forward
        self.activation = {v: k for k, v in ACTIVATIONS.items() if k}[d.activation]
        self.als_t = d.als_t

    @property
    def handle(self):
        return self._h

    def close(self):
        if self._h:
            load().dyra_layer_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def export(self) -> dict:
        """Host float64 copies of W_hat, W_res, P, R0 and the static factors."""
        d, m, r = self.d, self.m, self.r
        out = dict(W_hat=np.zeros((d, m)), W_res=np.zeros((d, m)), P=np.zeros((d, r)),
                   R0=np.zeros((r, m)))
        _check(load().dyra_export(self._h, out["W_hat"].ctypes.data, out["W_res"].ctypes.data,
                                  out["P"].ctypes.data, out["R0"].ctypes.data), "dyra_export")
        out["F1"], out["F2"] = _factor_arrays(self.kind, d, m, self.k)
        _check(load().dyra_export_factors(self._h, out["F1"].ctypes.data, out["F2"].ctypes.data),
               "dyra_export_factors")
        return out

    def workspace_size(self, batch: int, n: int) -> int:
        out = ctypes.c_size_t()
        _check(load().dyra_workspace_size(self._h, batch, n, ctypes.byref(out)),
               "dyra_workspace_size")
        return out.value

    def workspace_tensor(self, batch: int, n: int, which: str):
        off, ld = ctypes.c_size_t(), ctypes.c_int()
        _check(load().dyra_workspace_tensor(self._h, batch, n, BUFFERS[which], ctypes.byref(off),
                                            ctypes.byref(ld)), "dyra_workspace_tensor")
        return off.value, ld.value

    def kernel_names(self):
        return [load().dyra_kernel_name(self._h, i).decode()
                for i in range(self.kernels_per_forward)]


def _factor_arrays(kind, d, m, k, blast_t=0):
    if kind == "lowrank":
        return np.zeros((d, k)), np.zeros((k, m))
    if kind == "blast":
        return np.zeros((k, d // k, blast_t)), np.zeros((k, m // k, blast_t))
    return np.zeros((k, d // k, k)), np.zeros((k, k, m // k))


def _args(W, b, kind, k, r, R0, F1, F2, ridge, solver, ns_iters, dtype, device, fit_threads,
          calib=None, input_aware=None, activation=None, als_t=0.0, blast_t=0, F3=None):
    W = _f64(W)
    d, m = W.shape
    keep = dict(W=W, b=_f64(b, (m,)) if b is not None else None,
                R0=_f64(R0, (r, m)) if R0 is not None else None, F1=_f64(F1), F2=_f64(F2),
                F3=_f64(F3),
                calib=_f64(calib) if calib is not None else None)
    if keep["calib"] is not None and (keep["calib"].ndim != 2 or keep["calib"].shape[1] != d):
        raise ValueError(f"calib must be [n_calib, {d}]")
    args = PrepareArgs(W=_ptr(keep["W"]), b=_ptr(keep["b"]), d=d, m=m, kind=KINDS[kind], k=k, r=r,
                       R0=_ptr(keep["R0"]), F1=_ptr(keep["F1"]), F2=_ptr(keep["F2"]),
                       ridge=float(ridge), solver=SOLVERS[solver], ns_iters=ns_iters,
                       dtype=DTYPES[dtype], device=device, fit_threads=fit_threads,
                       calib=_ptr(keep["calib"]),
                       n_calib=0 if keep["calib"] is None else keep["calib"].shape[0],
                       input_aware=INPUT_AWARE[input_aware], activation=ACTIVATIONS[activation],
                       als_t=float(als_t), blast_t=int(blast_t), F3=_ptr(keep["F3"]))
    return args, keep


def prepare(W, b=None, kind: str = "lowrank", k: int = 0, r: int = 8, R0=None, F1=None, F2=None,
            ridge: float = 0.0, solver: str = "auto", ns_iters: int = 0, dtype: str = "bf16",
            device: int = 0, fit_threads: int = 0, calib=None, input_aware=None,
            activation=None, als_t: float = 0.0, blast_t: int = 0, F3=None) -> Layer:
    """dyra_prepare: offline fit, residual, R0, P and upload (synchronous). input_aware
    ("diag" or "cholesky") fits the static branch on the calibration rows `calib` [N, d];
    activation="gelu" applies GELU to the layer's output; als_t (1, 1.5, 2, ...) sets the
    number of ALS iterations of the correction; kind="blast" takes k = blocks per side,
    blast_t = the rank of every block's middle matrix and (optionally) F1/F2/F3 = U/V/S."""
    args, keep = _args(W, b, kind, k, r, R0, F1, F2, ridge, solver, ns_iters, dtype, device,
                       fit_threads, calib, input_aware, activation, als_t, blast_t, F3)
    h = ctypes.c_void_p()
    _check(load().dyra_prepare(ctypes.byref(args), ctypes.byref(h)), "dyra_prepare")
    del keep
    return Layer(h)


def fit(W, b=None, kind: str = "lowrank", k: int = 0, r: int = 8, R0=None, F1=None, F2=None,
        fit_threads: int = 0, calib=None, input_aware=None, blast_t: int = 0, F3=None) -> dict:
    """dyra_fit: the offline step on the host only; returns float64 arrays."""
    args, keep = _args(W, b, kind, k, r, R0, F1, F2, 0.0, "auto", 0, "bf16", 0, fit_threads,
                       calib, input_aware, None, 0.0, blast_t, F3)
    d, m = keep["W"].shape
    out = dict(W_hat=np.zeros((d, m)), W_res=np.zeros((d, m)), P=np.zeros((d, r)),
               R0=np.zeros((r, m)))
    out["F1"], out["F2"] = _factor_arrays(kind, d, m, k, blast_t)
    st = load().dyra_fit(ctypes.byref(args), *[out[key].ctypes.data for key in
                                                ("W_hat", "W_res", "P", "R0", "F1", "F2")])
    _check(st, "dyra_fit")
    return out


def _torch_dtype(layer):
    import torch
    return torch.bfloat16 if layer.dtype == "bf16" else torch.float32


def new_workspace(layer: Layer, batch: int, n: int):
    import torch
    nbytes = layer.workspace_size(batch, n)
    return torch.empty(max(nbytes, 256), dtype=torch.uint8, device=f"cuda:{layer.device}")


def _check_io(layer, X, Y):
    import torch
    if not (X.is_cuda and X.is_contiguous() and X.dtype == _torch_dtype(layer)):
        raise ValueError("X must be a contiguous CUDA tensor in the layer's dtype")
    if X.dim() != 3 or X.shape[2] != layer.d:
        raise ValueError(f"X must be [batch, n, {layer.d}]")
    if Y is None:
        Y = torch.empty((X.shape[0], X.shape[1], layer.m), dtype=X.dtype, device=X.device)
    elif not (Y.is_cuda and Y.is_contiguous() and Y.dtype == X.dtype and
              tuple(Y.shape) == (X.shape[0], X.shape[1], layer.m)):
        raise ValueError("Y must be a contiguous CUDA tensor [batch, n, m] in the layer's dtype")
    return Y


def linear_forward(layer: Layer, X, Y=None, workspace=None, stream=None):
    """dyra_linear_forward: enqueues the forward on `stream` (default: torch's current stream)."""
    Y = _check_io(layer, X, Y)
    batch, n = X.shape[0], X.shape[1]
    if workspace is None:
        workspace = new_workspace(layer, batch, n)
    st = load().dyra_linear_forward(layer.handle, ctypes.c_void_p(X.data_ptr()), batch, n,
                                    ctypes.c_void_p(Y.data_ptr()),
                                    ctypes.c_void_p(workspace.data_ptr()), workspace.numel(),
                                    _stream_handle(stream))
    _check(st, "dyra_linear_forward")
    return Y


def mlp_forward(fc1: Layer, fc2: Layer, X, H=None, Y=None, workspace=None, stream=None):
    """dyra_mlp_forward: H = fc1(X) (with fc1's activation), Y = fc2(H)."""
    import torch
    H = _check_io(fc1, X, H)
    Y = _check_io(fc2, H, Y)
    batch, n = X.shape[0], X.shape[1]
    if workspace is None:
        nbytes = max(fc1.workspace_size(batch, n), fc2.workspace_size(batch, n), 256)
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=f"cuda:{fc1.device}")
    st = load().dyra_mlp_forward(fc1.handle, fc2.handle, ctypes.c_void_p(X.data_ptr()), batch, n,
                                 ctypes.c_void_p(H.data_ptr()), ctypes.c_void_p(Y.data_ptr()),
                                 ctypes.c_void_p(workspace.data_ptr()), workspace.numel(),
                                 _stream_handle(stream))
    _check(st, "dyra_mlp_forward")
    return Y


def linear_forward_static(layer: Layer, X, Y=None, stream=None):
    """dyra_linear_forward_static: the forward with the library's static device scratch
    (no workspace argument, no device allocation by the library)."""
    Y = _check_io(layer, X, Y)
    st = load().dyra_linear_forward_static(layer.handle, ctypes.c_void_p(X.data_ptr()),
                                           X.shape[0], X.shape[1], ctypes.c_void_p(Y.data_ptr()),
                                           _stream_handle(stream))
    _check(st, "dyra_linear_forward_static")
    return Y


def linear_forward_host(layer: Layer, X_host, Y_host, X_dev, Y_dev, workspace, stream=None):
    """dyra_linear_forward_host: host X/Y (pinned torch CPU tensors), device staging buffers."""
    batch, n = X_host.shape[0], X_host.shape[1]
    st = load().dyra_linear_forward_host(layer.handle, ctypes.c_void_p(X_host.data_ptr()), batch,
                                         n, ctypes.c_void_p(Y_host.data_ptr()),
                                         ctypes.c_void_p(X_dev.data_ptr()),
                                         ctypes.c_void_p(Y_dev.data_ptr()),
                                         ctypes.c_void_p(workspace.data_ptr()), workspace.numel(),
                                         _stream_handle(stream))
    _check(st, "dyra_linear_forward_host")
    return Y_host


def linear_forward_profiled(layer: Layer, X, Y, workspace, events, stream=None) -> int:
    """dyra_linear_forward_profiled: `events` = torch.cuda.Event(enable_timing=True) objects,
    at least 2 * kernels_per_forward; events[2i] and events[2i + 1] bracket kernel i on the
    stream it runs on. Returns how many were recorded."""
    for e in events:           # torch creates the CUDA event lazily, on first record
        if e.cuda_event == 0:
            e.record()
    arr = (ctypes.c_void_p * len(events))(*[ctypes.c_void_p(e.cuda_event) for e in events])
    rec = ctypes.c_int()
    st = load().dyra_linear_forward_profiled(layer.handle, ctypes.c_void_p(X.data_ptr()),
                                             X.shape[0], X.shape[1], ctypes.c_void_p(Y.data_ptr()),
                                             ctypes.c_void_p(workspace.data_ptr()),
                                             workspace.numel(), _stream_handle(stream), arr,
                                             len(events), ctypes.byref(rec))
    _check(st, "dyra_linear_forward_profiled")
    return rec.value


def selftest_bounded_wait(limit_us: int, status_words, stream=None) -> int:
    """dyra_selftest_bounded_wait: runs the failure-path probe (a bounded wait that runs out)
    and returns its status code (TIMEOUT = 6 is the designed outcome). status_words: a CUDA
    tensor of at least 8 bytes; its first two int32 words receive the status counters."""
    if status_words.numel() * status_words.element_size() < 8:
        raise ValueError("status_words needs at least two 32-bit words")
    return load().dyra_selftest_bounded_wait(int(limit_us), ctypes.c_void_p(status_words.data_ptr()),
                                            _stream_handle(stream))


def workspace_status(layer: Layer, workspace, stream=None):
    """dyra_workspace_status: (not_spd_samples, timeouts); synchronises the stream."""
    a, b = ctypes.c_int(), ctypes.c_int()
    load().dyra_workspace_status(layer.handle, ctypes.c_void_p(workspace.data_ptr()),
                                 _stream_handle(stream), ctypes.byref(a), ctypes.byref(b))
    return a.value, b.value


def workspace_view(layer: Layer, workspace, batch: int, n: int, which: str, shape, dtype):
    """A torch view of an intermediate in the workspace (for per-kernel checks)."""
    import torch
    off, _ = layer.workspace_tensor(batch, n, which)
    count = int(np.prod(shape))
    esize = torch.empty((), dtype=dtype).element_size()
    return workspace[off:off + count * esize].view(dtype).view(*shape)
