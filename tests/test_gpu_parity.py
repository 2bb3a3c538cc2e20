"""GPU parity of the DyRA forward against the fp64 oracle, through the C ABI.

Every case runs the library's kernels on seeded synthetic inputs and compares with the
oracle on the same values: relative Frobenius error <= 1e-5 for fp32 layers and <= 2e-2
for bf16 layers, and the approximation error E = ||Y - b - XW|| / ||XW|| within 2% of the
oracle's. The library receives the oracle's static factors and R0, so singular-vector
signs and near-ties cannot confound the comparison (the library's own fit is checked
separately, on the host and in test_library_fit_end_to_end).
"""
import numpy as np
import pytest

import oracle as O
import workloads as WL
from gpu_util import (BF16_TOL, e_close, make_layer, oracle_solver, rel, to_device, to_host,
                      tol, weights_and_prep)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    import input_adaptive_rank_dyra_b300 as dy
    dy.load()
    yield


def _run(layer, X, dtype, ws=None):
    import torch
    import input_adaptive_rank_dyra_b300 as dy
    Xd = to_device(X, dtype)
    if ws is None:
        ws = dy.new_workspace(layer, X.shape[0], X.shape[1])
    Y = dy.linear_forward(layer, Xd, workspace=ws)
    torch.cuda.synchronize()
    return Y, ws


def _check_forward(cfg, X, W, b, prep, layer, Y, ridge=0.0):
    Yg = to_host(Y)
    Yo = O.forward(X, prep, ridge=ridge, solver=oracle_solver(layer), ns_iters=layer.ns_iters)
    err = rel(Yg, Yo)
    assert err <= tol(cfg), f"{cfg.name}: relative error {err:.3e} > {tol(cfg):.0e}"
    e_gpu = O.approximation_error(Yg, X, W, b)
    e_or = O.approximation_error(Yo, X, W, b)
    assert e_close(e_gpu, e_or), f"{cfg.name}: E gpu {e_gpu:.5f} vs oracle {e_or:.5f}"
    return err


# ---------------------------------------------------------------------------- reduced sizes

REDUCED = [("c1", None, None), ("c2", 3, None), ("c2", 2, 61), ("c3_fc1", 2, None),
           ("c3_fc2", 2, 300), ("c4", 2, None), ("c4", 3, 130), ("c5", 1, 1100),
           ("c6", 2, None), ("c6", 3, 100)]


@pytest.mark.parametrize("name,batch,n", REDUCED)
def test_forward_matches_oracle(name, batch, n):
    cfg = WL.reduced(WL.get_config(name), batch=batch, n=n)
    W, b, prep = weights_and_prep(name)
    X = WL.make_inputs(cfg)
    layer = make_layer(cfg, prep, W, b)
    Y, ws = _run(layer, X, cfg.dtype)
    _check_forward(cfg, X, W, b, prep, layer, Y)
    import input_adaptive_rank_dyra_b300 as dy
    assert dy.workspace_status(layer, ws) == (0, 0)


@pytest.mark.parametrize("name", ["c1", "c2", "c4"])
def test_intermediates_match_oracle(name):
    """Each kernel's output in the workspace: [XU | L], G, C, G^-1, then G^-1 C (bf16) or
    B = C W_res (fp32), and R = G^-1 C W_res."""
    import torch
    import input_adaptive_rank_dyra_b300 as dy
    cfg = WL.reduced(WL.get_config(name), batch=None if name == "c1" else 2,
                     n=300 if name == "c4" else None)
    W, b, prep = weights_and_prep(name)
    X = WL.make_inputs(cfg)
    layer = make_layer(cfg, prep, W, b)
    Y, ws = _run(layer, X, cfg.dtype)
    _, inter = O.forward(X, prep, keep=True)
    B_, n, d, m, k, r = cfg.batch, cfg.n, cfg.d, cfg.m, cfg.k, cfg.r
    t = tol(cfg)
    bf = cfg.dtype == "bf16"
    ft = torch.bfloat16 if bf else torch.float32
    _, ldT = layer.workspace_tensor(B_, n, "T")
    T = to_host(dy.workspace_view(layer, ws, B_, n, "T", (B_, n, ldT), ft))
    if cfg.kind == "monarch":
        # the static columns hold Zp[:, c*nb + a] = (X BD1)[:, a*nb + c]
        nb = k
        B1 = prep["F1"]
        Z = np.einsum("bnai,aic->bnac", X.reshape(B_, n, nb, d // nb), B1)
        assert rel(T[:, :, :d], Z.transpose(0, 1, 3, 2).reshape(B_, n, d)) <= t
        k = d
    else:
        XU = X @ prep["F1"]
        assert rel(T[:, :, :k], XU) <= t
    Lo = np.stack(inter["L"])
    Go = np.stack(inter["G"])
    Gi_o = np.linalg.inv(Go)
    gdt = torch.float32 if bf else torch.float64
    G = to_host(dy.workspace_view(layer, ws, B_, n, "G", (B_, r, r), gdt))
    assert rel(G, Go) <= t
    Gi = to_host(dy.workspace_view(layer, ws, B_, n, "GINV", (B_, r, r), ft if bf else gdt))
    assert rel(Gi, Gi_o) <= t
    if bf:   # C^T [batch, d, r], fp32
        C = to_host(dy.workspace_view(layer, ws, B_, n, "C", (B_, d, r), torch.float32))
        C = C.transpose(0, 2, 1)
    else:
        C = to_host(dy.workspace_view(layer, ws, B_, n, "C", (B_, r, d), ft))
    assert rel(C, np.stack(inter["C"])) <= t
    kl = ldT - r   # first L column of T
    assert rel(T[:, :, kl:kl + r], Lo) <= t
    if bf:
        # the solve runs on C before the residual product: C~ = G^-1 C, then R = C~ W_res
        Cs = to_host(dy.workspace_view(layer, ws, B_, n, "CS", (B_, r, d), ft))
        assert rel(Cs, Gi_o @ np.stack(inter["C"])) <= t
    else:
        Bm = to_host(dy.workspace_view(layer, ws, B_, n, "B", (B_, r, m), ft))
        assert rel(Bm, np.stack(inter["B"])) <= t
    R = to_host(dy.workspace_view(layer, ws, B_, n, "R", (B_, r, m), ft))
    assert rel(R, np.stack(inter["R"])) <= t


# ---------------------------------------------------------------------------- edge cases

# (batch, n): token counts around the 128-row tile and the 256-row CTA-pair unit. With more
# than one sample and n not a multiple of 256 the output GEMM tiles the flat batch * n rows,
# so a unit can hold the tail of one sample and the head of the next (or, for n < 128,
# parts of up to five samples); 256 and 512 keep the per-sample tiles.
TOKEN_CASES = [(2, 1), (2, 5), (2, 64), (2, 127), (2, 128), (2, 129), (2, 200), (7, 70),
               (5, 100), (3, 256), (4, 600), (2, 512)]


@pytest.mark.parametrize("batch,n", TOKEN_CASES)
def test_token_counts_spanning_tiles(batch, n):
    cfg = WL.reduced(WL.get_config("c2"), batch=batch, n=n)
    W, b, prep = weights_and_prep("c2")
    X = WL.make_inputs(cfg)
    layer = make_layer(cfg, prep, W, b)
    Y, _ = _run(layer, X, cfg.dtype)
    Yg = to_host(Y)
    Yo = O.forward(X, prep)
    assert rel(Yg, Yo) <= BF16_TOL
    # every sample on its own: a wrong segment would corrupt one sample's rows only
    for s in range(batch):
        assert rel(Yg[s], Yo[s]) <= BF16_TOL, f"sample {s}"


@pytest.mark.parametrize("name", ["c1", "c2"])
def test_zero_sample_falls_back_to_static(name):
    """An all-zero sample has L = 0, so L^T L is singular: R = 0, Y = static branch + b = b,
    and the sample is counted in the status word."""
    import input_adaptive_rank_dyra_b300 as dy
    cfg = WL.reduced(WL.get_config(name), batch=3, n=min(WL.get_config(name).n, 150))
    W, b, prep = weights_and_prep(name)
    X = WL.make_inputs(cfg)
    X[1] = 0.0
    layer = make_layer(cfg, prep, W, b)
    Y, ws = _run(layer, X, cfg.dtype)
    assert dy.workspace_status(layer, ws) == (1, 0)
    Yg = to_host(Y)
    bias = b.astype(np.float32)
    if cfg.dtype == "bf16":
        bias = WL.round_to_bf16(bias)
    assert np.array_equal(Yg[1], np.broadcast_to(bias, Yg[1].shape))
    Yo = O.forward(X, prep)
    keep = [0, 2]
    assert rel(Yg[keep], Yo[keep]) <= tol(cfg)


@pytest.mark.parametrize("name", ["c1", "c2"])
def test_ridge(name):
    cfg = WL.reduced(WL.get_config(name), batch=2)
    W, b, prep = weights_and_prep(name)
    X = WL.make_inputs(cfg)
    _, inter = O.forward(X, prep, keep=True)
    ridge = 0.5 * float(np.mean([np.trace(g) for g in inter["G"]])) / cfg.r
    layer = make_layer(cfg, prep, W, b, ridge=ridge)
    Y, _ = _run(layer, X, cfg.dtype)
    Yg = to_host(Y)
    Yo = O.forward(X, prep, ridge=ridge)
    assert rel(Yg, Yo) <= tol(cfg)
    assert rel(Yg, Yo) < rel(Yg, O.forward(X, prep))    # closer to the ridge solution


@pytest.mark.parametrize("name", ["c1", "c3_fc1"])
def test_newton_schulz_solver_matches_oracle_mirror(name):
    """The Newton-Schulz path (forced at r <= 64) against the oracle's NS iteration."""
    cfg = WL.reduced(WL.get_config(name), batch=2, n=None if name == "c1" else 500)
    W, b, prep = weights_and_prep(name)
    X = WL.make_inputs(cfg)
    for iters in (3, 8):
        layer = make_layer(cfg, prep, W, b, solver="newton_schulz", ns_iters=iters)
        assert layer.solver == "newton_schulz"
        Y, _ = _run(layer, X, cfg.dtype)
        Yo = O.forward(X, prep, solver="newton_schulz", ns_iters=iters)
        assert rel(to_host(Y), Yo) <= tol(cfg)


def test_batch_zero_is_noop():
    import input_adaptive_rank_dyra_b300 as dy
    import torch
    cfg = WL.get_config("c2")
    W, b, prep = weights_and_prep("c2")
    layer = make_layer(cfg, prep, W, b)
    X = torch.empty((0, 10, cfg.d), dtype=torch.bfloat16, device="cuda")
    Y = dy.linear_forward(layer, X)
    assert Y.shape == (0, 10, cfg.m)


def test_deterministic_and_host_path_identical():
    """Two forwards give the same bits; the host-buffer entry point gives the same bits."""
    import torch
    import input_adaptive_rank_dyra_b300 as dy
    cfg = WL.reduced(WL.get_config("c2"), batch=4)
    W, b, prep = weights_and_prep("c2")
    X = WL.make_inputs(cfg)
    layer = make_layer(cfg, prep, W, b)
    Y1, ws = _run(layer, X, cfg.dtype)
    Y2, _ = _run(layer, X, cfg.dtype, ws)
    assert torch.equal(Y1.view(torch.int16), Y2.view(torch.int16))
    Xh = to_device(X, "bf16").cpu().pin_memory()
    Yh = torch.empty(Y1.shape, dtype=torch.bfloat16).pin_memory()
    Xs = torch.empty_like(Xh, device="cuda")
    Ys = torch.empty(Y1.shape, dtype=torch.bfloat16, device="cuda")
    dy.linear_forward_host(layer, Xh, Yh, Xs, Ys, ws)
    torch.cuda.synchronize()
    assert torch.equal(Yh.view(torch.int16), Y1.cpu().view(torch.int16))


def test_host_path_in_sample_groups_identical():
    """A batch large enough (84 MB of X and Y) for the host-buffer entry point to cut it into
    eight groups of one sample, whose copies and forwards overlap on three streams: the same
    bits as the device-buffer forward of the whole batch, and the status words clean."""
    import torch
    import input_adaptive_rank_dyra_b300 as dy
    cfg = WL.reduced(WL.get_config("c3_fc1"), batch=8)
    W, b, prep = weights_and_prep("c3_fc1")
    X = WL.make_inputs(cfg)
    layer = make_layer(cfg, prep, W, b)
    Y1, ws = _run(layer, X, cfg.dtype)
    Xh = to_device(X, "bf16").cpu().pin_memory()
    Yh = torch.full(Y1.shape, float("nan"), dtype=torch.bfloat16).pin_memory()
    Xs = torch.empty_like(Xh, device="cuda")
    Ys = torch.empty(Y1.shape, dtype=torch.bfloat16, device="cuda")
    for _ in range(2):
        dy.linear_forward_host(layer, Xh, Yh, Xs, Ys, ws)
        torch.cuda.synchronize()
        assert torch.equal(Yh.view(torch.int16), Y1.cpu().view(torch.int16))
        assert dy.workspace_status(layer, ws) == (0, 0)


def test_profiled_forward_records_every_kernel():
    import torch
    import input_adaptive_rank_dyra_b300 as dy
    cfg = WL.reduced(WL.get_config("c2"), batch=2)
    W, b, prep = weights_and_prep("c2")
    X = WL.make_inputs(cfg)
    layer = make_layer(cfg, prep, W, b)
    Xd = to_device(X, "bf16")
    ws = dy.new_workspace(layer, cfg.batch, cfg.n)
    Y = torch.empty((cfg.batch, cfg.n, cfg.m), dtype=torch.bfloat16, device="cuda")
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2 * layer.kernels_per_forward)]
    got = dy.linear_forward_profiled(layer, Xd, Y, ws, ev)
    torch.cuda.synchronize()
    assert got == 2 * layer.kernels_per_forward
    times = [ev[2 * i].elapsed_time(ev[2 * i + 1]) for i in range(layer.kernels_per_forward)]
    assert all(t > 0 for t in times)
    assert rel(to_host(Y), O.forward(X, prep)) <= BF16_TOL
    assert len(layer.kernel_names()) == layer.kernels_per_forward


def test_library_fit_end_to_end():
    """dyra_prepare fitting the static branch and R0 itself: the output is invariant to the
    fit's gauge, so it matches the oracle run on its own fit."""
    import input_adaptive_rank_dyra_b300 as dy
    cfg = WL.reduced(WL.get_config("c2"), batch=2)
    W, b, prep = weights_and_prep("c2")
    X = WL.make_inputs(cfg)
    layer = dy.prepare(W, b, kind="lowrank", k=cfg.k, r=cfg.r, dtype="bf16", device=0)
    Y, _ = _run(layer, X, "bf16")
    assert rel(to_host(Y), O.forward(X, prep)) <= BF16_TOL


# ---------------------------------------------------------------------------- full sizes

FULL = ["c2", "c3_fc1", "c3_fc2", "c4", "c5", "c6"]


@pytest.mark.parametrize("name", FULL)
def test_full_size_sampled_rows(name):
    """The full workload in the launch configuration the benchmark times; the oracle forms
    every per-sample factor (L, G, C, B, R use all tokens) but only sampled output rows."""
    import input_adaptive_rank_dyra_b300 as dy
    cfg = WL.get_config(name)
    W, b, prep = weights_and_prep(name)
    X = WL.make_inputs(cfg)
    layer = make_layer(cfg, prep, W, b)
    Y, ws = _run(layer, X, cfg.dtype)
    assert dy.workspace_status(layer, ws) == (0, 0)
    Yg = to_host(Y)
    rng = np.random.default_rng(1234)
    per = 48
    rows = [np.sort(rng.choice(cfg.n, size=min(per, cfg.n), replace=False))
            for _ in range(cfg.batch)]
    # always include the first and last token of each sample (tile edges)
    rows = [np.unique(np.concatenate([r_, [0, cfg.n - 1]])) for r_ in rows]
    Yo = O.forward(X, prep, solver=oracle_solver(layer), ns_iters=layer.ns_iters, rows=rows)
    Ys = np.concatenate([Yg[s][rows[s]] for s in range(cfg.batch)])
    Yo = np.concatenate(Yo)
    err = rel(Ys, Yo)
    assert err <= BF16_TOL, f"{name}: {err:.3e}"
    Xs = np.concatenate([X[s][rows[s]] for s in range(cfg.batch)])
    e_gpu = O.approximation_error(Ys, Xs, W, b)
    e_or = O.approximation_error(Yo, Xs, W, b)
    assert e_close(e_gpu, e_or), f"{name}: E gpu {e_gpu:.5f} vs oracle {e_or:.5f}"
    if layer.solver == "newton_schulz":
        # the iteration must also reach the explicit least-squares solution's error
        Yc = np.concatenate(O.forward(X, prep, solver="cholesky", rows=rows))
        e_chol = O.approximation_error(Yc, Xs, W, b)
        assert e_close(e_gpu, e_chol), f"{name}: E gpu {e_gpu:.5f} vs explicit {e_chol:.5f}"
