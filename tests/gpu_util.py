"""Helpers shared by the GPU tests: move seeded inputs to the device, run the layer through
the C ABI, and compare against the fp64 oracle."""
from __future__ import annotations

import functools

import numpy as np

import oracle as O
import workloads as WL

BF16_TOL = 2e-2     # relative Frobenius error allowed for bf16 layers
F32_TOL = 1e-5      # ... and for fp32 layers
E_REL_TOL = 0.02    # |E_gpu - E_oracle| <= 2% of E_oracle


def tol(cfg) -> float:
    return F32_TOL if cfg.dtype == "f32" else BF16_TOL


@functools.lru_cache(maxsize=None)
def weights_and_prep(name: str):
    """(W, b, oracle preparation) of a named layer, computed once per test session."""
    cfg = WL.get_config(name)
    W, b = WL.make_weights(cfg)
    k = (cfg.k, cfg.blast_t) if cfg.kind == "blast" else cfg.k
    prep = O.prepare(W, b, cfg.kind, k, cfg.r)
    return W, b, prep


def to_device(X: np.ndarray, dtype: str):
    import torch
    if dtype == "bf16":
        bits = WL.bf16_bits(X).view(np.int16)
        return torch.from_numpy(np.ascontiguousarray(bits)).view(torch.bfloat16).cuda()
    return torch.from_numpy(np.ascontiguousarray(X, dtype=np.float32)).cuda()


def to_host(T) -> np.ndarray:
    return T.float().cpu().numpy().astype(np.float64)


def make_layer(cfg, prep, W, b, **kw):
    import input_adaptive_rank_dyra_b300 as dy
    args = dict(kind=cfg.kind, k=cfg.k, r=cfg.r, F1=prep["F1"], F2=prep["F2"], R0=prep["R0"],
                dtype=cfg.dtype, device=0, solver=cfg.solver, ns_iters=cfg.ns_iters)
    if cfg.kind == "blast":
        args.update(blast_t=cfg.blast_t, F3=prep["F3"])
    args.update(kw)
    return dy.prepare(W, b, **args)


def oracle_solver(layer) -> str:
    return "cholesky" if layer.solver == "cholesky" else "newton_schulz"


def rel(a, b) -> float:
    return O.relative_frobenius(np.asarray(a, dtype=np.float64), np.asarray(b, dtype=np.float64))


def e_close(e_gpu: float, e_or: float) -> bool:
    return abs(e_gpu - e_or) <= E_REL_TOL * e_or
