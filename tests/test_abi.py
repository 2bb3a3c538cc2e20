"""CPU tests of the C ABI: the library loads, exports every entry point the header declares,
rejects bad arguments without touching a device, and its host-side offline fit matches the
oracle. No compute call runs on a GPU here."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle as O
import workloads as WL
from input_adaptive_rank_dyra_b300 import dyra as D

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _header_functions():
    text = open(os.path.join(ROOT, "include", "dyra.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dyra_[a-z_0-9]+)\s*\(", text)))


def test_library_exports_every_declared_function():
    lib = D.load()
    declared = _header_functions()
    assert "dyra_prepare" in declared and "dyra_linear_forward" in declared
    for name in declared:
        assert hasattr(lib, name), name
    assert set(declared) <= set(D.EXPORTED)
    assert lib.dyra_abi_version() == 3


def test_status_strings():
    lib = D.load()
    for code in range(9):
        assert lib.dyra_status_string(code)
    assert lib.dyra_status_string(0) == b"ok"


def _args(W, **kw):
    W = np.ascontiguousarray(W, dtype=np.float64)
    a = D.PrepareArgs()
    a.W = W.ctypes.data_as(D._c_double_p)
    a.d, a.m = W.shape
    a.kind, a.k, a.r = 0, 4, 2
    a.dtype = 1
    for key, val in kw.items():
        setattr(a, key, val)
    return a, W


@pytest.mark.parametrize("bad", [
    dict(d=0), dict(r=0), dict(k=-1), dict(k=40), dict(ridge=-1.0), dict(kind=7), dict(dtype=9),
    dict(solver=9),
])
def test_prepare_rejects_bad_arguments(bad):
    lib = D.load()
    W = np.random.default_rng(0).standard_normal((32, 48))
    a, keep = _args(W, **bad)
    h = ctypes.c_void_p()
    assert lib.dyra_prepare(ctypes.byref(a), ctypes.byref(h)) == 1   # INVALID_ARG
    assert not h.value


def test_prepare_rejects_null_and_unsupported():
    lib = D.load()
    h = ctypes.c_void_p()
    assert lib.dyra_prepare(None, ctypes.byref(h)) == 1
    W = np.random.default_rng(0).standard_normal((32, 48))
    a, keep = _args(W, r=6)          # the bf16 kernels need r % 8 == 0
    assert lib.dyra_prepare(ctypes.byref(a), ctypes.byref(h)) == 2
    a, keep = _args(W, r=8, solver=1, k=0)   # fine for validation; a device is then needed
    assert lib.dyra_prepare(ctypes.byref(a), ctypes.byref(h)) in (0, 8)


def test_forward_rejects_bad_arguments_without_device():
    lib = D.load()
    assert lib.dyra_linear_forward(None, None, 1, 1, None, None, 0, None) == 1
    assert lib.dyra_workspace_size(None, 1, 1, None) == 1
    assert lib.dyra_workspace_status(None, None, None, None, None) == 1
    assert lib.dyra_kernel_name(None, 0) is None
    # the failure-path self-test checks its arguments before any CUDA call
    assert lib.dyra_selftest_bounded_wait(1000, None, None) == 1
    assert lib.dyra_selftest_bounded_wait(0, ctypes.c_void_p(4096), None) == 1
    assert lib.dyra_selftest_bounded_wait(3000000, ctypes.c_void_p(4096), None) == 1


def test_fit_lowrank_matches_oracle():
    cfg = WL.get_config("c2")
    W, b = WL.make_weights(cfg)
    f = D.fit(W, kind="lowrank", k=cfg.k, r=cfg.r)
    p = O.prepare(W, b, "lowrank", cfg.k, cfg.r)
    scale = np.abs(W).max()
    assert np.abs(f["W_hat"] - p["W_hat"]).max() < 1e-9 * scale
    assert np.abs(f["W_res"] - p["W_res"]).max() < 1e-9 * scale
    # R0 and P are fixed up to an r x r rotation; the projector and P R0 are not
    assert np.allclose(f["R0"].T @ f["R0"], p["R0"].T @ p["R0"], atol=1e-8)
    assert np.abs(f["P"] @ f["R0"] - p["P"] @ p["R0"]).max() < 1e-9 * scale


def test_fit_with_supplied_r0_and_factors():
    rng = np.random.default_rng(3)
    W = rng.standard_normal((40, 56))
    p = O.prepare(W, np.zeros(56), "lowrank", 6, 5)
    R0 = rng.standard_normal((5, 56))
    f = D.fit(W, kind="lowrank", k=6, r=5, R0=R0, F1=p["F1"], F2=p["F2"])
    assert np.allclose(f["W_hat"], p["W_hat"], atol=1e-12)
    assert np.allclose(f["P"], O.projection(p["W_res"], R0), atol=1e-10)


def test_fit_monarch_matches_oracle():
    cfg = WL.get_config("c4")
    W, b = WL.make_weights(cfg)
    f = D.fit(W, kind="monarch", k=cfg.k, r=cfg.r)
    p = O.prepare(W, b, "monarch", cfg.k, cfg.r)
    scale = np.abs(W).max()
    assert np.abs(f["W_hat"] - p["W_hat"]).max() < 1e-9 * scale
    assert np.abs(f["P"] @ f["R0"] - p["P"] @ p["R0"]).max() < 1e-8 * scale


@pytest.mark.parametrize("mode", ["diag", "cholesky"])
def test_fit_input_aware_matches_oracle(mode):
    """The library's input-aware static fit (host fp64, its own eigensolver and Cholesky)
    against the oracle's, on the DINOv3 fc1 weights with calibration rows of the same
    per-sample-covariance recipe: W_hat, W_res and the projector P R0 agree."""
    cfg = WL.reduced(WL.get_config("c3_fc1"))
    W, b = WL.make_weights(cfg)
    Xc = WL.make_calibration(cfg, 3000)
    f = D.fit(W, kind="lowrank", k=cfg.k, r=cfg.r, calib=Xc, input_aware=mode)
    U, V = O.input_aware_factors(W, cfg.k, Xc, mode)
    p = O.prepare(W, b, "lowrank", cfg.k, cfg.r, factors=(U, V))
    scale = np.abs(W).max()
    assert np.abs(f["W_hat"] - p["W_hat"]).max() < 1e-8 * scale
    assert np.abs(f["P"] @ f["R0"] - p["P"] @ p["R0"]).max() < 1e-7 * scale
    plain = O.prepare(W, b, "lowrank", cfg.k, cfg.r)
    # the fit is input-aware: a smaller output error on the calibration rows than plain TSVD
    assert (np.linalg.norm(Xc @ p["W_res"]) < np.linalg.norm(Xc @ plain["W_res"]))


def test_fit_r0_from_rank_deficient_residual():
    """Static factors given, R0 not: R0 comes from the SVD of W_res, which for a truncated-SVD
    W_hat has d - k exactly-zero singular values (a cluster of zero eigenvalues in the Gram
    matrix that the eigensolver must still deflate)."""
    cfg = WL.get_config("c2")
    W, b = WL.make_weights(cfg)
    p = O.prepare(W, b, "lowrank", cfg.k, cfg.r)
    f = D.fit(W, kind="lowrank", k=cfg.k, r=cfg.r, F1=p["F1"], F2=p["F2"])
    scale = np.abs(W).max()
    assert np.abs(f["P"] @ f["R0"] - p["P"] @ p["R0"]).max() < 1e-8 * scale


def test_fit_input_aware_rejects_bad_calibration():
    W = np.random.default_rng(5).standard_normal((16, 24))
    with pytest.raises(D.DyraError):      # fewer rows than features: covariance singular
        D.fit(W, kind="lowrank", k=3, r=2, calib=np.ones((4, 16)), input_aware="cholesky")
    with pytest.raises(D.DyraError):      # no calibration rows
        D.fit(W, kind="lowrank", k=3, r=2, input_aware="diag")


def test_fit_blast_matches_oracle():
    """The library's BLAST fit (host fp64, its own SVDs; 10 alternating sweeps from the same
    start) against the oracle's on the BLAST workload's weights: the same W_hat (each step
    depends only on the subspaces, not on their bases)."""
    cfg = WL.get_config("c6")
    W, b = WL.make_weights(cfg)
    f = D.fit(W, kind="blast", k=cfg.k, r=cfg.r, blast_t=cfg.blast_t)
    p = O.prepare(W, b, "blast", (cfg.k, cfg.blast_t), cfg.r)
    scale = np.abs(W).max()
    assert np.abs(f["W_hat"] - p["W_hat"]).max() < 1e-8 * scale
    assert np.abs(f["P"] @ f["R0"] - p["P"] @ p["R0"]).max() < 1e-7 * scale
    # and the structure is BLAST: every block row of W_hat has rank <= t
    t, nb, pb = cfg.blast_t, cfg.k, cfg.d // cfg.k
    for i in range(nb):
        assert np.linalg.matrix_rank(f["W_hat"][i * pb:(i + 1) * pb], tol=1e-9 * scale) <= t


def test_fit_rejects_rank_deficient_r0():
    W = np.random.default_rng(4).standard_normal((20, 30))
    R0 = np.zeros((3, 30))
    R0[0, 0] = R0[1, 0] = R0[2, 1] = 1.0
    with pytest.raises(D.DyraError):
        D.fit(W, kind="lowrank", k=2, r=3, R0=R0)
