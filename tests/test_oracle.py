"""Pins for the fp64 oracle: facts that the pages and the mathematics fix, checked
against routines other than the ones the oracle itself calls.

Each test names the passage it pins. A plausible slip in the oracle (a dropped
(R0 R0^T)^-1, a transposed factor, a wrong Monarch index, a missing bias, an off-by-one
in Newton-Schulz) fails at least one of them.
"""
import numpy as np
import pytest

import oracle as O
import workloads as WL


def _rng(seed):
    return np.random.default_rng(seed)


def _orth(rng, rows, cols):
    q, _ = np.linalg.qr(rng.standard_normal((rows, cols)))
    return q


def _top_left_projector(W, p):
    """Projector onto W's top-p left singular subspace, via eigh of W W^T
    (a different LAPACK route from the oracle's SVD)."""
    w, v = np.linalg.eigh(W @ W.T)
    top = v[:, np.argsort(w)[::-1][:p]]
    return top @ top.T


def _small_case(seed=0, n=40, d=24, m=36, k=5, r=4, batch=3):
    rng = _rng(seed)
    W = rng.standard_normal((d, m)) * (np.arange(1, d + 1) ** -0.5)[:, None]
    b = rng.standard_normal(m) * 0.1
    X = rng.standard_normal((batch, n, d)) * np.linspace(3.0, 0.3, d)[None, None, :]
    return W, b, X, k, r


# -------------------------------------------------------------------- static fit

def test_tsvd_is_frobenius_optimal_rank_k():
    """Appendix B (truncated SVD is the best rank-k approximation in Frobenius norm):
    ||W - W_hat||_F^2 equals the sum of the trailing eigenvalues of W^T W."""
    W, _, _, k, _ = _small_case()
    U, V = O.tsvd_factors(W, k)
    What = O.lowrank_dense(U, V)
    lam = np.sort(np.linalg.eigvalsh(W.T @ W))[::-1]
    assert np.linalg.matrix_rank(What) == k
    assert np.isclose(np.linalg.norm(W - What) ** 2, lam[k:].sum(), rtol=1e-10)
    # W_hat is the projection of W onto its top-k left singular subspace
    assert np.allclose(What, _top_left_projector(W, k) @ W, atol=1e-11)
    # even split of the singular values: U^T U == V V^T (both diag(S_k))
    assert np.allclose(U.T @ U, V @ V.T, atol=1e-11)


def _planted_monarch(rng, nb, bi, bo):
    """Dense matrix built entry by entry from W[(a,i),(c,j)] = B1[a][i,c] B2[c][a,j]."""
    B1 = rng.standard_normal((nb, bi, nb))
    B2 = rng.standard_normal((nb, nb, bo))
    W = np.zeros((nb * bi, nb * bo))
    for a in range(nb):
        for i in range(bi):
            for c in range(nb):
                for j in range(bo):
                    W[a * bi + i, c * bo + j] = B1[a][i, c] * B2[c][a, j]
    return W, B1, B2


def test_monarch_dense_matches_index_form():
    """Appendix B / blog structured-methods section: block-diagonal . stride permutation .
    block-diagonal equals the per-block rank-1 index form."""
    rng = _rng(1)
    W, B1, B2 = _planted_monarch(rng, 4, 3, 5)
    assert np.allclose(O.monarch_dense(B1, B2), W, atol=1e-13)


def test_monarch_fit_recovers_planted_monarch():
    rng = _rng(2)
    W, _, _ = _planted_monarch(rng, 4, 4, 4)
    B1, B2 = O.monarch_factors(W, 4)
    assert np.linalg.norm(W - O.monarch_dense(B1, B2)) < 1e-12 * np.linalg.norm(W)


def test_monarch_fit_is_blockwise_optimal():
    """The fit's error equals the sum over blocks of the non-leading eigenvalues of each
    block's Gram matrix (best rank-1 per block)."""
    rng = _rng(3)
    nb, bi, bo = 4, 4, 6
    W = rng.standard_normal((nb * bi, nb * bo))
    B1, B2 = O.monarch_factors(W, nb)
    err = np.linalg.norm(W - O.monarch_dense(B1, B2)) ** 2
    tail = 0.0
    for a in range(nb):
        for c in range(nb):
            blk = W[a * bi:(a + 1) * bi, c * bo:(c + 1) * bo]
            lam = np.sort(np.linalg.eigvalsh(blk @ blk.T))[::-1]
            tail += lam[1:].sum()
    assert np.isclose(err, tail, rtol=1e-10)


# -------------------------------------------------------------------- BLAST fit

def _planted_blast(rng, nb, p, q, t):
    U = rng.standard_normal((nb, p, t))
    V = rng.standard_normal((nb, q, t))
    S = rng.standard_normal((nb, nb, t, t))
    W = np.zeros((nb * p, nb * q))
    for i in range(nb):                    # entry by entry: sum over the middle matrix
        for j in range(nb):
            for a in range(p):
                for c in range(q):
                    W[i * p + a, j * q + c] = sum(U[i, a, x] * S[i, j, x, y] * V[j, c, y]
                                                  for x in range(t) for y in range(t))
    return W, U, V, S


def test_blast_dense_matches_index_form():
    """Appendix B / blog structured-methods section: W_hat[(i,a),(j,c)] =
    sum_{x,y} U[i][a,x] S[i,j][x,y] V[j][c,y]."""
    rng = _rng(30)
    W, U, V, S = _planted_blast(rng, 3, 4, 5, 2)
    assert np.allclose(O.blast_dense(U, V, S), W, atol=1e-12)


def test_blast_fit_recovers_planted_blast():
    """A matrix that is exactly BLAST (nb = 3, t = 2) is reproduced: each block row has rank
    t, so the SVD start spans the true bases and the middle matrices are exact."""
    rng = _rng(31)
    W, _, _, _ = _planted_blast(rng, 3, 6, 5, 2)
    for sweeps in (0, 3):
        U, V, S = O.blast_factors(W, 3, 2, sweeps=sweeps)
        assert np.linalg.norm(W - O.blast_dense(U, V, S)) < 1e-10 * np.linalg.norm(W)


def test_blast_fit_error_never_increases_and_middles_are_optimal():
    """Each step is an exact minimiser, so the reconstruction error does not increase with
    the sweeps; the middle matrices are the least-squares optimum for their bases (the block
    residual is orthogonal to both bases), checked against lstsq on the vectorised block."""
    rng = _rng(32)
    W = rng.standard_normal((12, 16))
    errs = [np.linalg.norm(W - O.blast_dense(*O.blast_factors(W, 4, 2, sweeps=s)))
            for s in (0, 1, 2, 5, 20)]
    assert all(errs[i + 1] <= errs[i] * (1 + 1e-12) for i in range(len(errs) - 1))
    assert errs[-1] < errs[0]
    U, V, S = O.blast_factors(W, 4, 2, sweeps=5)
    p, q = 3, 4
    for i in range(4):
        for j in range(4):
            Wij = W[i * p:(i + 1) * p, j * q:(j + 1) * q]
            A = np.kron(U[i], V[j])          # vec(U S V^T) = (U kron V) vec(S), row-major vec
            s_ls = np.linalg.lstsq(A, Wij.reshape(-1), rcond=None)[0]
            assert np.allclose(S[i, j].reshape(-1), s_ls, atol=1e-10)


def test_blast_forward_exact_when_residual_rank_at_most_r():
    """BLAST branch end to end: W = BLAST + A R0 with rank(A) <= r and the planted factors gives
    Y = X W + b."""
    rng = _rng(33)
    Wb, U, V, S = _planted_blast(rng, 2, 6, 5, 2)
    r = 2
    A = rng.standard_normal((12, r))
    R0 = _orth(rng, 10, r).T
    W = Wb + A @ R0
    b = rng.standard_normal(10)
    X = rng.standard_normal((2, 20, 12))
    prep = O.prepare(W, b, "blast", (2, 2), r, R0=R0, factors=(U, V, S))
    assert np.allclose(prep["W_res"], A @ R0, atol=1e-11)
    assert np.allclose(O.forward(X, prep), X @ W + b, atol=1e-9 * np.abs(X @ W).max())


# -------------------------------------------------------------------- input-aware fit

def _correlated_calibration(rng, N, d):
    """Rows with a strongly anisotropic, correlated covariance."""
    Q = _orth(rng, d, d)
    return (rng.standard_normal((N, d)) * np.geomspace(5.0, 0.05, d)[None, :]) @ Q.T


def test_input_aware_cholesky_is_optimal_on_calibration_rows():
    """Appendix B input-aware decomposition with S the Cholesky factor of the calibration
    covariance: the output error on the calibration rows equals the smallest any rank-k W_hat
    can reach, the sum of the trailing eigenvalues of W^T X^T X W (Eckart-Young on S^T W),
    here computed by eigh of that matrix directly; the plain truncated SVD does worse."""
    rng = _rng(20)
    d, m, k, N = 16, 24, 5, 200
    W = rng.standard_normal((d, m))
    Xc = _correlated_calibration(rng, N, d)
    U, V = O.input_aware_factors(W, k, Xc, "cholesky")
    What = U @ V
    assert np.linalg.matrix_rank(What) == k
    err = np.linalg.norm(Xc @ (W - What)) ** 2
    lam = np.sort(np.linalg.eigvalsh(W.T @ (Xc.T @ Xc) @ W))[::-1]
    assert np.isclose(err, lam[k:].sum(), rtol=1e-9)
    Up, Vp = O.tsvd_factors(W, k)
    assert err < np.linalg.norm(Xc @ (W - Up @ Vp)) ** 2


def test_input_aware_reduces_to_tsvd_for_isotropic_calibration():
    """With X^T X = c I (isotropic calibration) both scalings are multiples of the identity,
    and the input-aware W_hat is the plain truncated SVD."""
    rng = _rng(21)
    d, m, k = 12, 20, 4
    W = rng.standard_normal((d, m))
    Xc = 3.0 * _orth(rng, 60, d)
    Up, Vp = O.tsvd_factors(W, k)
    for mode in ("cholesky", "diag"):
        U, V = O.input_aware_factors(W, k, Xc, mode)
        assert np.allclose(U @ V, Up @ Vp, atol=1e-10)


def test_input_aware_diag_scaling_weights_channels():
    """Diagonal mode: S = diag(channel rms). For calibration rows with independent channels
    of known scales, W_hat is the best rank-k fit of W in the norm weighted by those scales:
    it equals diag(1/s) TSVD_k(diag(s) W), checked against the weighted problem solved by
    eigh, and its calibration error is below the plain truncated SVD's."""
    rng = _rng(22)
    d, m, k, N = 10, 14, 3, 4000
    scales = np.geomspace(4.0, 0.1, d)
    Xc = rng.standard_normal((N, d)) * scales[None, :]
    W = rng.standard_normal((d, m))
    U, V = O.input_aware_factors(W, k, Xc, "diag")
    s = np.sqrt(np.mean(Xc * Xc, axis=0))
    Ws = s[:, None] * W
    w, vecs = np.linalg.eigh(Ws @ Ws.T)
    top = vecs[:, np.argsort(w)[::-1][:k]]
    assert np.allclose(U @ V, (top @ top.T @ Ws) / s[:, None], atol=1e-10)
    Up, Vp = O.tsvd_factors(W, k)
    assert np.linalg.norm(Xc @ (W - U @ V)) < np.linalg.norm(Xc @ (W - Up @ Vp))


def test_input_aware_fit_ignores_calibration_scale():
    """Scaling every calibration row by the same factor leaves W_hat unchanged."""
    rng = _rng(23)
    W = rng.standard_normal((12, 16))
    Xc = _correlated_calibration(rng, 100, 12)
    for mode in ("cholesky", "diag"):
        U1, V1 = O.input_aware_factors(W, 4, Xc, mode)
        U2, V2 = O.input_aware_factors(W, 4, 7.0 * Xc, mode)
        assert np.allclose(U1 @ V1, U2 @ V2, atol=1e-10)


# -------------------------------------------------------------------- residual / R0 / P

def test_residual_split_is_exact():
    """Blog residual-split section: X W = X W_hat + X W_res."""
    W, _, X, k, r = _small_case()
    prep = O.prepare(W, np.zeros(W.shape[1]), "lowrank", k, r)
    XU = X @ prep["F1"]
    lhs = XU @ prep["F2"] + X @ prep["W_res"]
    assert np.allclose(lhs, X @ W, atol=1e-12)


def test_r0_is_next_singular_block_for_lowrank():
    """2.3 / blog one-step section: for a low-rank W_hat the residual's top-r right singular
    vectors span W's right singular vectors k+1..k+r."""
    W, _, _, k, r = _small_case()
    prep = O.prepare(W, np.zeros(W.shape[1]), "lowrank", k, r)
    w, v = np.linalg.eigh(W.T @ W)
    v = v[:, np.argsort(w)[::-1]]
    span = v[:, k:k + r]
    R0 = prep["R0"]
    assert np.allclose(R0 @ R0.T, np.eye(r), atol=1e-12)
    assert np.allclose(span @ span.T, R0.T @ R0, atol=1e-9)


def test_projection_inverts_r0_gram():
    """The L-update with R fixed: if W_res = A R0 for any full-row-rank R0 (not
    orthonormal), then P = A exactly. A dropped (R0 R0^T)^-1 fails here."""
    rng = _rng(4)
    A = rng.standard_normal((10, 3))
    R0 = rng.standard_normal((3, 14)) * 3.0
    assert np.allclose(O.projection(A @ R0, R0), A, atol=1e-12)


# -------------------------------------------------------------------- the online step

@pytest.mark.parametrize("ridge", [0.0, 0.7])
def test_r_is_least_squares_solution(ridge):
    """Blog rank-r objective section: with L fixed, R minimises ||X W_res - L R||_F^2
    (+ ridge ||R||_F^2, 2.2). Brute force: LAPACK lstsq on the stacked system."""
    W, b, X, k, r = _small_case(seed=5)
    prep = O.prepare(W, b, "lowrank", k, r)
    _, inter = O.forward(X, prep, ridge=ridge, keep=True)
    for s in range(X.shape[0]):
        L = X[s] @ prep["P"]
        target = X[s] @ prep["W_res"]
        A = np.vstack([L, np.sqrt(ridge) * np.eye(r)])
        rhs = np.vstack([target, np.zeros((r, W.shape[1]))])
        R_ls = np.linalg.lstsq(A, rhs, rcond=None)[0]
        assert np.allclose(inter["R"][s], R_ls, atol=1e-10)


def test_normal_equations_hold():
    """Residual of the R-update is orthogonal to range(L): L^T (X W_res - L R) = 0."""
    for name in ("c1",):
        cfg = WL.get_config(name)
        W, b = WL.make_weights(cfg)
        X = WL.make_inputs(cfg)
        prep = O.prepare(W, b, cfg.kind, cfg.k, cfg.r)
        _, inter = O.forward(X, prep, keep=True)
        for s in range(X.shape[0]):
            L, R = inter["L"][s], inter["R"][s]
            e = X[s] @ prep["W_res"] - L @ R
            scale = np.linalg.norm(L) * np.linalg.norm(X[s] @ prep["W_res"])
            assert np.linalg.norm(L.T @ e) <= 1e-10 * scale


def test_output_is_static_plus_bias_plus_correction():
    """Y = X W_hat + b + L R with the bias added exactly once (W_hat taken from the factors)."""
    W, b, X, k, r = _small_case(seed=6)
    prep = O.prepare(W, b, "lowrank", k, r)
    Y, inter = O.forward(X, prep, keep=True)
    for s in range(X.shape[0]):
        corr = inter["L"][s] @ inter["R"][s]
        assert np.allclose(Y[s] - (X[s] @ prep["F1"]) @ prep["F2"] - corr, b[None, :], atol=1e-12)


def test_exact_when_residual_rank_at_most_r():
    """If rank(W_res) <= r and R0 spans its row space, L R = X W_res, so Y = X W + b."""
    rng = _rng(7)
    d, m, k, r = 20, 30, 4, 3
    W = _orth(rng, d, k + r) @ np.diag(np.linspace(5, 1, k + r)) @ _orth(rng, m, k + r).T
    b = rng.standard_normal(m)
    X = rng.standard_normal((2, 25, d))
    prep = O.prepare(W, b, "lowrank", k, r)
    Y = O.forward(X, prep)
    assert np.allclose(Y, X @ W + b, atol=1e-10)
    # non-orthonormal R0 spanning the same rows gives the same output
    M = rng.standard_normal((r, r)) + 3 * np.eye(r)
    prep2 = O.prepare(W, b, "lowrank", k, r, R0=M @ prep["R0"])
    assert np.allclose(O.forward(X, prep2), X @ W + b, atol=1e-9)


def test_proposition1_isotropic_input():
    """Proposition 1 (2.3, Appendix C): with X^T X = c I, one-step DyRA equals the static
    rank-(k+r) truncated SVD and R equals R0."""
    rng = _rng(8)
    n, d, m, k, r = 64, 24, 40, 5, 6
    W = rng.standard_normal((d, m)) * (np.arange(1, d + 1) ** -0.7)[:, None]
    c = 2.5
    X = (np.sqrt(c) * _orth(rng, n, d))[None]
    prep = O.prepare(W, np.zeros(m), "lowrank", k, r)
    Y, inter = O.forward(X, prep, keep=True)
    assert np.allclose(inter["R"][0], prep["R0"], atol=1e-9)
    assert np.allclose(Y[0], X[0] @ (_top_left_projector(W, k + r) @ W), atol=1e-9)


def test_lr_error_above_eckart_young_bound_and_als_monotone():
    """E.3: ALS error is bounded below by the optimal rank-r error of X W_res (SVD of the
    residual product) and does not increase with more ALS iterations."""
    W, _, X, k, r = _small_case(seed=9, n=50)
    prep = O.prepare(W, np.zeros(W.shape[1]), "lowrank", k, r)
    Xs = X[0]
    target = Xs @ prep["W_res"]
    lam = np.sort(np.linalg.eigvalsh(target.T @ target))[::-1]
    bound = np.sqrt(max(lam[r:].sum(), 0.0))
    errs = []
    for t in (1, 1.5, 2, 3, 5, 40):
        L, R = O.als_factors(Xs, prep["W_res"], prep["R0"], t)
        errs.append(np.linalg.norm(target - L @ R))
    _, inter = O.forward(X[:1], prep, keep=True)
    assert np.isclose(np.linalg.norm(target - inter["L"][0] @ inter["R"][0]), errs[0], rtol=1e-10)
    assert all(e >= bound * (1 - 1e-12) for e in errs)
    assert all(errs[i + 1] <= errs[i] * (1 + 1e-12) for i in range(len(errs) - 1))
    assert errs[-1] <= bound * (1 + 1e-3)


def test_als_half_steps_satisfy_their_normal_equations():
    """E.3 / Figure 9 ALS variants: after t = 1.5 (L, R, L) the last L-update is the
    least-squares L for the R it used, (X W_res - L R) R^T = 0; after t = 2 the last R-update
    satisfies L^T (X W_res - L R) = 0; t = 1 reproduces forward()."""
    W, b, X, k, r = _small_case(seed=25, n=50)
    prep = O.prepare(W, b, "lowrank", k, r)
    Xs = X[0]
    target = Xs @ prep["W_res"]
    L1, R1 = O.als_factors(Xs, prep["W_res"], prep["R0"], 1)
    L15, R15 = O.als_factors(Xs, prep["W_res"], prep["R0"], 1.5)
    assert np.allclose(R15, R1, atol=1e-12)     # t = 1.5 keeps the t = 1 right factor
    scale = np.linalg.norm(target) * np.linalg.norm(R15)
    assert np.abs((target - L15 @ R15) @ R15.T).max() < 1e-10 * scale
    L2, R2 = O.als_factors(Xs, prep["W_res"], prep["R0"], 2)
    assert np.abs(L2.T @ (target - L2 @ R2)).max() < 1e-10 * np.linalg.norm(L2) * np.linalg.norm(target)
    assert np.allclose(O.forward_als(X, prep, 1), O.forward(X, prep), atol=1e-10)
    # forward_als and als_factors are written separately; they agree for every t
    for t, (Lt, Rt) in ((1.5, (L15, R15)), (2, (L2, R2))):
        Yt = O.forward_als(X[:1], prep, t)
        assert np.allclose(Yt[0], Xs @ prep["W_hat"] + b + Lt @ Rt, atol=1e-9)
    # with the Newton-Schulz solver run to convergence the same result comes out
    Yns = O.forward_als(X[:1], prep, 2, solver="newton_schulz", ns_iters=40)
    assert np.allclose(Yns[0], Xs @ prep["W_hat"] + b + L2 @ R2, atol=1e-8)


def test_gauge_invariance_of_r0():
    """Rotating or sign-flipping R0's rows leaves L R (hence Y) unchanged."""
    rng = _rng(10)
    W, b, X, k, r = _small_case(seed=10)
    prep = O.prepare(W, b, "lowrank", k, r)
    Q = _orth(rng, r, r)
    Q[:, 0] *= -1
    prep2 = O.prepare(W, b, "lowrank", k, r, R0=Q @ prep["R0"])
    assert np.allclose(O.forward(X, prep), O.forward(X, prep2), atol=1e-10)


def test_zero_sample_falls_back_to_static_branch():
    """Degenerate case: an all-zero sample gives L = 0 and G = 0 (not SPD); its output is
    the bias (static branch of a zero input)."""
    W, b, X, k, r = _small_case(seed=11)
    X = X.copy()
    X[1] = 0.0
    prep = O.prepare(W, b, "lowrank", k, r)
    Y, inter = O.forward(X, prep, keep=True)
    assert inter["ok"] == [True, False, True]
    assert np.allclose(Y[1], b[None, :], atol=0)


def test_rows_subset_matches_full_forward():
    W, b, X, k, r = _small_case(seed=12)
    prep = O.prepare(W, b, "lowrank", k, r)
    Y = O.forward(X, prep)
    rows = [np.array([0, 7, 39]), np.array([3]), np.array([5, 6])]
    Ys = O.forward(X, prep, rows=rows)
    for s in range(3):
        assert np.allclose(Ys[s], Y[s][rows[s]], atol=1e-12)


# -------------------------------------------------------------------- Newton-Schulz

def test_newton_schulz_closed_form():
    """With X0 = alpha I, I - G_hat X_t = (I - alpha G_hat)^(2^t) exactly, so on G_hat's
    eigenvalues mu: x_t(mu) = (1 - (1 - alpha mu)^(2^t)) / mu."""
    rng = _rng(13)
    A = rng.standard_normal((40, 12)) * np.linspace(3, 0.5, 12)[None, :]
    G = A.T @ A
    dinv = 1 / np.sqrt(np.diag(G))
    Gh = G * dinv[:, None] * dinv[None, :]
    mu, V = np.linalg.eigh(Gh)
    alpha = 1.0 / np.max(np.abs(Gh).sum(axis=1))
    for t in (1, 2, 5, 8):
        x = (1 - (1 - alpha * mu) ** (2 ** t)) / mu
        expect = (V * x[None, :]) @ V.T * dinv[:, None] * dinv[None, :]
        assert np.allclose(O.newton_schulz_inverse(G, t), expect, rtol=1e-9, atol=1e-12)


def test_newton_schulz_converges_to_inverse():
    rng = _rng(14)
    A = rng.standard_normal((300, 32))
    G = A.T @ A
    assert np.allclose(O.newton_schulz_inverse(G, 30), np.linalg.inv(G), rtol=1e-11, atol=1e-14)
    B = rng.standard_normal((32, 7))
    R, ok = O.solve_right_factor(G, B, "newton_schulz", 30)
    assert ok and np.allclose(R, np.linalg.solve(G, B), rtol=1e-10, atol=1e-12)


# -------------------------------------------------------------------- MLP block

def test_gelu_table_values():
    """GELU(x) = x Phi(x) at points where the standard normal CDF is tabulated:
    Phi(1) = 0.8413447460685429, Phi(2) = 0.9772498680518208, Phi(0) = 1/2; and
    GELU(x) - GELU(-x) = x (Phi(x) + Phi(-x) = 1)."""
    assert O.gelu(np.array([1.0]))[0] == pytest.approx(0.8413447460685429, rel=1e-14)
    assert O.gelu(np.array([-1.0]))[0] == pytest.approx(-(1 - 0.8413447460685429), rel=1e-13)
    assert O.gelu(np.array([2.0]))[0] == pytest.approx(2 * 0.9772498680518208, rel=1e-14)
    assert O.gelu(np.array([0.0]))[0] == 0.0
    x = np.linspace(-6, 6, 97)
    assert np.allclose(O.gelu(x) - O.gelu(-x), x, atol=1e-14)
    assert np.allclose(O.gelu(np.array([40.0, -40.0])), [40.0, 0.0], atol=1e-12)


def test_mlp_block_exact_when_both_residuals_have_rank_at_most_r():
    """Both layers exact (rank(W_res) <= r, R0 spanning it): the DyRA MLP block equals the
    dense GELU(X W1 + b1) W2 + b2."""
    rng = _rng(24)
    d, hdim, m, k, r = 12, 20, 10, 3, 2
    W1 = _orth(rng, d, k + r) @ np.diag(np.linspace(4, 1, k + r)) @ _orth(rng, hdim, k + r).T
    W2 = _orth(rng, hdim, k + r) @ np.diag(np.linspace(3, 1, k + r)) @ _orth(rng, m, k + r).T
    b1, b2 = rng.standard_normal(hdim), rng.standard_normal(m)
    X = rng.standard_normal((2, 30, d))
    p1 = O.prepare(W1, b1, "lowrank", k, r)
    p2 = O.prepare(W2, b2, "lowrank", k, r)
    ref = O.gelu(X @ W1 + b1) @ W2 + b2
    assert np.allclose(O.mlp_forward(X, p1, p2), ref, atol=1e-9)


# -------------------------------------------------------------------- metric and workloads

def test_relative_frobenius_hand_value():
    """The parity metric ||a - b||_F / ||b||_F on values worked out by hand:
    a - b = [[0, 0], [0, -1]] and ||b||_F^2 = 1 + 4 + 9 + 25 = 39, so the value is 1/sqrt(39).
    With a = 2 b the two argument orders give 1 and 1/2, so a swapped numerator and
    denominator, or a missing square root (1/39, or 1 and 1/4), fails."""
    a = np.array([[1.0, 2.0], [3.0, 4.0]])
    b = np.array([[1.0, 2.0], [3.0, 5.0]])
    assert O.relative_frobenius(a, b) == pytest.approx(0.16012815380508713, rel=1e-15)
    assert O.relative_frobenius(2 * b, b) == pytest.approx(1.0, rel=1e-15)
    assert O.relative_frobenius(b, 2 * b) == pytest.approx(0.5, rel=1e-15)
    assert O.relative_frobenius(b, b) == 0.0


def test_monarch_forward_exact_when_residual_rank_at_most_r():
    """Monarch branch end to end (Appendix B structure; blog rank-r objective and one-step
    sections): with W = Monarch(B1, B2) + A R0, rank(A) <= r, the static factors (B1, B2) and
    any R0 spanning the residual's row space, the residual is A R0 exactly, so P = A (R0
    orthonormal), L = X A, R = R0 and Y = X W + b. A wrong permutation index, a dropped
    static term or a transposed block would leave a residual the rank-r correction cannot
    absorb."""
    rng = _rng(16)
    nb, bi, bo, r = 4, 3, 5, 3
    Wm, B1, B2 = _planted_monarch(rng, nb, bi, bo)
    d, m = nb * bi, nb * bo
    A = rng.standard_normal((d, r))
    R0 = _orth(rng, m, r).T
    W = Wm + A @ R0
    b = rng.standard_normal(m)
    X = rng.standard_normal((2, 30, d))
    prep = O.prepare(W, b, "monarch", nb, r, R0=R0, factors=(B1, B2))
    assert np.allclose(prep["W_res"], A @ R0, atol=1e-12)
    assert np.allclose(prep["P"], A, atol=1e-12)
    Y, inter = O.forward(X, prep, keep=True)
    assert np.allclose(Y, X @ W + b, atol=1e-10 * np.abs(X @ W).max())
    # the library-side convention: the residual rank-r term alone is X W_res
    for s in range(2):
        assert np.allclose(inter["L"][s] @ inter["R"][s], X[s] @ (A @ R0), atol=1e-10)
    # with R0 taken from the residual's own SVD (another basis of the same rows), the
    # output is the same
    prep2 = O.prepare(W, b, "monarch", nb, r, factors=(B1, B2))
    assert not np.allclose(prep2["R0"], R0, atol=1e-6)
    assert np.allclose(O.forward(X, prep2), X @ W + b, atol=1e-10 * np.abs(X @ W).max())


def test_approximation_error_metric():
    rng = _rng(15)
    X = rng.standard_normal((2, 5, 4))
    W = rng.standard_normal((4, 3))
    b = rng.standard_normal(3)
    assert O.approximation_error(X @ W + b, X, W, b) < 1e-15
    assert np.isclose(O.approximation_error(b + 0 * (X @ W), X, W, b), 1.0)


def test_c1_dyra_beats_static_truncation():
    """c1 end to end: the correction lowers the output error below the static rank-k fit,
    and Proposition 1's comparison point (static rank k+r) is beaten on anisotropic X."""
    cfg = WL.get_config("c1")
    W, b = WL.make_weights(cfg)
    X = WL.make_inputs(cfg)
    prep = O.prepare(W, b, cfg.kind, cfg.k, cfg.r)
    Y = O.forward(X, prep)
    e_dyra = O.approximation_error(Y, X, W, b)
    e_static = O.approximation_error(X @ prep["W_hat"] + b, X, W, b)
    U2, V2 = O.tsvd_factors(W, cfg.k + cfg.r)
    e_static_kr = O.approximation_error(X @ (U2 @ V2) + b, X, W, b)
    assert e_dyra < e_static_kr < e_static


def test_input_aware_scaling_hand_values():
    """The input-side transform on a 2 x 2 calibration matrix worked out by hand:
    X_cal = [[1, 2], [3, 4]] has channel mean squares 5 and 10, so diag gives
    diag(sqrt 5, sqrt 10); its covariance X_cal^T X_cal / 2 = [[5, 7], [7, 10]] has the lower
    Cholesky factor [[sqrt 5, 0], [7 / sqrt 5, sqrt(10 - 49 / 5)]]."""
    X = np.array([[1.0, 2.0], [3.0, 4.0]])
    S = O.input_aware_scaling(X, "diag")
    assert np.allclose(S, np.diag([np.sqrt(5.0), np.sqrt(10.0)]), atol=1e-15)
    L = O.input_aware_scaling(X, "cholesky")
    expect = np.array([[np.sqrt(5.0), 0.0], [7.0 / np.sqrt(5.0), np.sqrt(10.0 - 49.0 / 5.0)]])
    assert np.allclose(L, expect, atol=1e-14)
    with pytest.raises(ValueError):
        O.input_aware_scaling(X, "other")


def test_top_right_singular_subspace_and_energy():
    """R0 of a residual with a planted SVD: orthonormal rows spanning the top-r right singular
    subspace, and W_res R0^T R0 keeps exactly the top-r singular values' energy
    (Eckart-Young), whatever basis the SVD returns for that subspace."""
    rng = _rng(31)
    d, m, r = 12, 9, 3
    Q1, _ = np.linalg.qr(rng.standard_normal((d, m)))
    Q2, _ = np.linalg.qr(rng.standard_normal((m, m)))
    sv = np.array([9.0, 7.0, 5.0, 1.0, 0.8, 0.5, 0.3, 0.2, 0.1])
    W_res = Q1 @ np.diag(sv) @ Q2.T
    R0 = O.top_right_singular(W_res, r)
    assert R0.shape == (r, m)
    assert np.allclose(R0 @ R0.T, np.eye(r), atol=1e-12)
    top = Q2[:, :r]
    assert np.allclose(R0.T @ R0, top @ top.T, atol=1e-12)
    kept = np.linalg.norm(W_res @ R0.T @ R0) ** 2
    assert np.isclose(kept, np.sum(sv[:r] ** 2), rtol=1e-12)
