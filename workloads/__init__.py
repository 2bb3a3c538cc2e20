"""Seeded synthetic inputs for the DyRA linear layer.

This module only draws random numbers and rounds them to the storage type the
layer consumes. It holds none of the method's arithmetic (no static fit, no
residual, no least-squares step), so both the fp64 oracle and the CUDA path can
take their inputs from it without sharing any computation.

The five layer shapes follow the workloads the DyRA paper evaluates
("DyRA: Dynamic Residual Approximation for Efficient Matrix Multiplication in
DNNs", Appendix D: ViT-B/16 and ViT-L image models, DINOv3 dense prediction,
LLM prefill in Appendix E.1), scaled to one linear layer each. No dataset,
checkpoint or benchmark item is used: every tensor is drawn from a seeded
PCG64 stream.

Every sample of X is drawn from its own stream (seed, tensor id, sample index),
so a test that generates only the first few samples of a workload gets exactly
the rows that the full workload holds.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np
from scipy.linalg import solve_triangular

__all__ = ["LayerConfig", "CONFIGS", "get_config", "make_weights", "make_inputs",
           "make_calibration", "round_to_bf16", "bf16_bits", "reduced"]


@dataclasses.dataclass(frozen=True)
class LayerConfig:
    name: str
    batch: int
    n: int              # tokens per sample
    d: int              # input features (c1 in the paper's notation)
    m: int              # output features (c2)
    kind: str           # "lowrank" or "monarch"
    k: int              # static rank (low-rank) or number of Monarch blocks
    r: int              # residual (dynamic) rank
    dtype: str          # "f32" or "bf16": storage type of X, Y and the device factors
    seed: int
    w_recipe: str       # "planted" | "powerlaw"
    w_exponent: float   # sigma_i proportional to i^-w_exponent (powerlaw recipe)
    x_recipe: str       # "geometric" | "outliers" | "covariance" | "student_t"
    solver: str = "auto"
    ns_iters: int = 8
    als_t: float = 1.0  # ALS iterations of the correction (1: the one-step form)
    blast_t: int = 0    # BLAST: rank of every block's middle matrix (k = blocks per side)
    stream: int = 0     # distinguishes two layers that share a seed (fc1 / fc2)

    @property
    def tokens(self) -> int:
        return self.batch * self.n


CONFIGS = {
    # One fp32 layer: anisotropic X, a planted rank-8 component of strength 3 on top of
    # N(0, 1/d) noise; k = 16, r = 8.
    "c1": LayerConfig("c1_fp32_single_layer", 1, 64, 128, 256, "lowrank", 16, 8, "f32", 0,
                      "planted", 0.0, "geometric"),
    # ViT-B/16 MLP fc1: 64 images x 197 tokens, 768 -> 3072, k = 192, r = 32.
    "c2": LayerConfig("c2_vitb16_fc1", 64, 197, 768, 3072, "lowrank", 192, 32, "bf16", 2,
                      "powerlaw", 0.7, "outliers"),
    # DINOv3 ViT-L/16 at 512x512 (32x32 patches + cls + 4 registers = 1029 tokens).
    "c3_fc1": LayerConfig("c3_dinov3_vitl16_fc1", 16, 1029, 1024, 4096, "lowrank", 256, 64, "bf16", 3,
                          "powerlaw", 0.6, "covariance", stream=0),
    "c3_fc2": LayerConfig("c3_dinov3_vitl16_fc2", 16, 1029, 4096, 1024, "lowrank", 256, 64, "bf16", 3,
                          "powerlaw", 0.6, "covariance", stream=1),
    # Attention projection 1024 -> 1024 with a Monarch static branch of 32 blocks of 32x32.
    "c4": LayerConfig("c4_monarch32_attn_proj", 16, 1029, 1024, 1024, "monarch", 32, 64, "bf16", 4,
                      "powerlaw", 0.7, "outliers"),
    # BLAST static branch (4 x 4 blocks of 256 x 256, middle matrices of rank 64) plus the
    # correction on the attention-projection shape of c4; W and X drawn as in config 2.
    "c6": LayerConfig("c6_blast4x64_attn_proj", 16, 1029, 1024, 1024, "blast", 4, 64, "bf16", 6,
                      "powerlaw", 0.7, "outliers", blast_t=64),
    # LLM prefill MLP up-projection 4096 -> 12288, k = 1024, r = 256, Newton-Schulz (8 steps).
    "c5": LayerConfig("c5_prefill_mlp_up", 4, 2048, 4096, 12288, "lowrank", 1024, 256, "bf16", 5,
                      "powerlaw", 0.5, "student_t", solver="newton_schulz", ns_iters=8),
}


def get_config(name: str) -> LayerConfig:
    return CONFIGS[name]


def reduced(cfg: LayerConfig, batch: Optional[int] = None, n: Optional[int] = None) -> LayerConfig:
    """Same layer (same W, same per-sample X streams) with fewer samples or tokens."""
    return dataclasses.replace(cfg, batch=cfg.batch if batch is None else batch,
                               n=cfg.n if n is None else n)


# ----------------------------------------------------------------------------------
# storage rounding

def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round to bfloat16 (fp32 first, then round-to-nearest-even on the upper 16 bits);
    returns float64 values that are exactly representable in bf16."""
    return bf16_bits_to_f64(bf16_bits(x))


def bf16_bits(x: np.ndarray) -> np.ndarray:
    f = np.ascontiguousarray(x, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    nan = np.isnan(f)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    out = rounded.astype(np.uint16)
    if nan.any():
        out[nan] = 0x7FC0
    return out


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    u = bits.astype(np.uint32) << 16
    return u.view(np.float32).astype(np.float64)


# ----------------------------------------------------------------------------------
# random building blocks

def _rng(cfg: LayerConfig, *path: int) -> np.random.Generator:
    return np.random.default_rng([cfg.seed, cfg.stream, *path])


def _haar(rng: np.random.Generator, rows: int, cols: int) -> np.ndarray:
    """rows x cols matrix with orthonormal columns, Haar distributed (QR of a Gaussian
    with the signs of R's diagonal folded into Q)."""
    g = rng.standard_normal((rows, cols))
    if cols < 2048:
        q, rr = np.linalg.qr(g)
        q *= np.sign(np.diag(rr))[None, :]
        return q
    # Large bases: two Cholesky-QR passes (BLAS-3 only, several times faster than
    # Householder QR here). Both passes produce an upper-triangular factor with a
    # positive diagonal, so Q is the same Haar-distributed factor as above.
    q = g
    for _ in range(2):
        c = np.linalg.cholesky(q.T @ q)          # q^T q = c c^T, c lower triangular
        q = solve_triangular(c, q.T, lower=True, check_finite=False).T   # q <- q c^{-T}
    return q


_W_ID, _B_ID, _X_ID, _XCH_ID = 1, 2, 3, 4


def make_weights(cfg: LayerConfig):
    """Returns (W [d, m] float64, b [m] float64). The bias is stored in fp32 by the layer,
    so it is returned rounded to fp32."""
    rng = _rng(cfg, _W_ID)
    d, m = cfg.d, cfg.m
    if cfg.w_recipe == "planted":
        # N(0, 1/d) entries plus 3 * Qu Qv^T: eight directions of strength 3 planted
        # above a noise bulk whose singular values reach about 1 + sqrt(m/d) = 2.41.
        w = rng.standard_normal((d, m)) / math.sqrt(d)
        qu = _haar(rng, d, 8)
        qv = _haar(rng, m, 8)
        w += 3.0 * qu @ qv.T
    elif cfg.w_recipe == "powerlaw":
        p = min(d, m)
        q1 = _haar(rng, d, p)
        q2 = _haar(rng, m, p)
        sig = np.arange(1, p + 1, dtype=np.float64) ** (-cfg.w_exponent)
        sig *= math.sqrt(d * m * 0.02 ** 2 / float(np.sum(sig ** 2)))   # ||W||_F^2 = d m 0.02^2
        w = (q1 * sig[None, :]) @ q2.T
    else:
        raise ValueError(cfg.w_recipe)
    brng = _rng(cfg, _B_ID)
    if cfg.w_recipe == "planted":
        b = brng.normal(0.0, math.sqrt(0.01), size=m)   # N(0, 0.01): variance 0.01
    else:
        b = brng.normal(0.0, 0.02, size=m)
    b = b.astype(np.float32).astype(np.float64)
    return np.ascontiguousarray(w), b


def _outlier_channels(cfg: LayerConfig) -> np.ndarray:
    rng = _rng(cfg, _XCH_ID)
    count = int(round(0.01 * cfg.d))
    return np.sort(rng.choice(cfg.d, size=count, replace=False))


def _channel_scales(cfg: LayerConfig) -> np.ndarray:
    rng = _rng(cfg, _XCH_ID)
    return rng.uniform(0.1, 10.0, size=cfg.d)


def _sample(cfg: LayerConfig, s: int) -> np.ndarray:
    rng = _rng(cfg, _X_ID, s)
    n, d = cfg.n, cfg.d
    if cfg.x_recipe == "geometric":
        # columns scaled geometrically from 4 down to 0.25
        scale = 4.0 * 16.0 ** (-np.arange(d) / max(d - 1, 1))
        return rng.standard_normal((n, d)) * scale[None, :]
    if cfg.x_recipe == "outliers":
        x = rng.standard_normal((n, d))
        x[:, _outlier_channels(cfg)] *= 20.0
        return x
    if cfg.x_recipe == "covariance":
        # X_s = Z diag(sqrt(lambda)) Q_s^T: covariance eigenvalues lambda_i ~ 1/i (mean 1)
        # in a per-sample Haar eigenbasis.
        lam = 1.0 / np.arange(1, d + 1, dtype=np.float64)
        lam *= d / lam.sum()
        q = _haar(rng, d, d)
        z = rng.standard_normal((n, d))
        return (z * np.sqrt(lam)[None, :]) @ q.T
    if cfg.x_recipe == "student_t":
        return rng.standard_t(4.0, size=(n, d)) * _channel_scales(cfg)[None, :]
    raise ValueError(cfg.x_recipe)


_CALIB_BASE = 1_000_000   # sample indices of calibration draws (disjoint from the workload's)


def make_calibration(cfg: LayerConfig, rows: int) -> np.ndarray:
    """Calibration activations [rows, d] for an input-aware fit: the rows of fresh samples of
    the same recipe, drawn from streams no workload sample uses (float64; bf16-representable
    for bf16 layers, like the inputs)."""
    out, s = [], 0
    while sum(x.shape[0] for x in out) < rows:
        out.append(_sample(cfg, _CALIB_BASE + s))
        s += 1
    x = np.concatenate(out)[:rows]
    return round_to_bf16(x) if cfg.dtype == "bf16" else x.astype(np.float32).astype(np.float64)


def make_inputs(cfg: LayerConfig, samples: Optional[range] = None) -> np.ndarray:
    """X [len(samples), n, d] float64; for bf16 layers the values are bf16-representable
    (the layer's input is the bf16 tensor; the oracle reads the same values in fp64)."""
    idx = range(cfg.batch) if samples is None else samples
    x = np.stack([_sample(cfg, s) for s in idx]) if len(idx) else np.zeros((0, cfg.n, cfg.d))
    if cfg.dtype == "bf16":
        return round_to_bf16(x)
    return x.astype(np.float32).astype(np.float64)
