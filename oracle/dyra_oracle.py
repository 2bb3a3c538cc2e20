"""fp64 CPU oracle of the DyRA linear layer.

TEST INFRASTRUCTURE ONLY. The library (package ``input_adaptive_rank_dyra_b300``)
never imports, links or runs anything here and has no CPU fallback. Only the test
suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` use it.

It is a plain, slow, step-by-step restatement of what the pages define, in float64,
one sample at a time, with numpy/scipy library calls (SVD, Cholesky, matmul) as the
only building blocks. There is no blocking, fusion or reordering beyond what the
definitions state.

Sources, cited per function:
  [S] "DyRA: Dynamic Residual Approximation for Efficient Matrix Multiplication in DNNs"
      -- section-by-section summary page (paperlayer.ai): 2.2 Dynamic Residual
      Approximation, 2.3 Analysis of One-Step ALS (Proposition 1, cost), 2.4
      Implementation, Appendix B (structured matrices), Appendix C (proof of Prop. 1),
      E.3 (ALS convergence).
  [B] "DyRA：用输入相关的残差修正加速大模型的矩阵乘法" -- blog digest (nanless.github.io):
      section "静态分支与残差如何拆分" (static branch / residual split, the two equations
      W = W_hat + W_res and XW = X W_hat + X W_res), section "残差乘积的低秩优化目标是什么"
      (rank-r objective min ||X W_res - L R||_F^2 and the order of operations of the two
      ALS updates), section "一次迭代的近似形式与额外代价" (one-step form
      XW ~ X W_hat + L(1) R(1); R0 from the residual's singular vectors k+1..k+r), section
      "没有训练时离线准备和在线计算是什么" (offline preparation: R0 = top right singular
      vectors of W_res, projection precomputed once), section "已有结构化矩阵方法分工有何不同"
      (Monarch: block-diagonal, permutation, block-diagonal; fitted by truncated SVD of
      each block of the rearranged dense weight).

Readings taken where the pages are silent (the same list is kept with the design notes):
  * ridge: absolute lambda added to L^T L, default 0 (the pages use "a small ridge term"
    without a value);
  * projection P = W_res R0^T (R0 R0^T)^-1: the least-squares L-update with R = R0 fixed;
  * the singular values of the low-rank fit are split evenly: U = U_k sqrt(S_k),
    V = sqrt(S_k) V_k^T (Y does not depend on the split);
  * Monarch with nb blocks: W_hat[(a,i),(c,j)] = B1[a][i,c] * B2[c][a,j]; each
    (a,c) block of W gets its best rank-1 approximation;
  * BLAST with nb x nb blocks of rank t: block (i,j) = U[i] S[i,j] V[j]^T with a t x t middle
    matrix per block (the pages' "small middle matrix"), fitted by alternating exact
    minimisations from per-block-row and per-block-column truncated SVDs, a fixed number of
    sweeps;
  * Newton-Schulz: Jacobi scaling G_hat = D G D with D = diag(G)^-1/2, X0 = I/||G_hat||_inf,
    X_{t+1} = X_t (2I - G_hat X_t), G^-1 ~ D X_T D;
  * input-aware decomposition, written for the row-vector convention y = x W used here:
    W_hat = S^-T TSVD_k(S^T W), with S = diag(channel rms) or the lower Cholesky factor of the
    calibration covariance; R0 and P are then formed from W_res as for the plain fit;
  * one least-squares system per sample over all of its n tokens;
  * a sample whose G is not positive definite (e.g. an all-zero sample with lambda = 0)
    gets R = 0, i.e. its output is the static branch plus the bias.
"""
from __future__ import annotations

import numpy as np
import scipy.linalg as sla

__all__ = [
    "tsvd_factors", "lowrank_dense", "monarch_factors", "monarch_dense", "blast_factors",
    "blast_dense", "input_aware_scaling",
    "input_aware_factors", "residual",
    "top_right_singular", "projection", "prepare", "newton_schulz_inverse",
    "solve_right_factor", "forward", "als_factors", "forward_als", "gelu", "mlp_forward",
    "approximation_error",
    "relative_frobenius",
]


# ------------------------------------------------------------------------------------
# offline preparation

def tsvd_factors(W: np.ndarray, k: int):
    """Truncated SVD of W at rank k, returned as U (d x k) and V (k x m) with
    W_hat = U V the Frobenius-optimal rank-k approximation.
    [S] Appendix B (truncated SVD keeps the top components); [B] structured-methods section."""
    u, s, vt = np.linalg.svd(W, full_matrices=False)
    root = np.sqrt(s[:k])
    return u[:, :k] * root[None, :], root[:, None] * vt[:k]


def lowrank_dense(U: np.ndarray, V: np.ndarray) -> np.ndarray:
    return U @ V


def monarch_factors(W: np.ndarray, nb: int):
    """Monarch fit with nb blocks: B1 [nb, d/nb, nb] and B2 [nb, nb, m/nb].

    W_hat = blockdiag(B1[0..nb-1]) . (stride permutation) . blockdiag(B2[0..nb-1]); in
    index form W_hat[(a,i),(c,j)] = B1[a][i,c] B2[c][a,j], so every (a,c) block of the
    dense weight is a rank-1 outer product, and the fit takes the best rank-1 approximation
    (leading singular triplet) of each block.
    [S] Appendix B (Monarch: block-diagonal factors and a permutation); [B] structured-methods
    section (each block of the rearranged dense weight gets a truncated SVD)."""
    d, m = W.shape
    bi, bo = d // nb, m // nb
    if bi * nb != d or bo * nb != m:
        raise ValueError("Monarch needs d and m divisible by the block count")
    B1 = np.zeros((nb, bi, nb))
    B2 = np.zeros((nb, nb, bo))
    for a in range(nb):
        for c in range(nb):
            blk = W[a * bi:(a + 1) * bi, c * bo:(c + 1) * bo]
            u, s, vt = np.linalg.svd(blk)
            root = np.sqrt(s[0])
            B1[a][:, c] = root * u[:, 0]
            B2[c][a, :] = root * vt[0]
    return B1, B2


def monarch_dense(B1: np.ndarray, B2: np.ndarray) -> np.ndarray:
    """Dense W_hat = BD1 @ Pi @ BD2 (row-vector convention y = x W_hat).
    BD1 maps input (a,i) to intermediate (a,c) with block B1[a]; Pi sends intermediate
    (a,c) to (c,a); BD2 maps (c,a) to output (c,j) with block B2[c]."""
    nb, bi, _ = B1.shape
    bo = B2.shape[2]
    bd1 = sla.block_diag(*[B1[a] for a in range(nb)])            # (nb*bi) x (nb*nb)
    bd2 = sla.block_diag(*[B2[c] for c in range(nb)])            # (nb*nb) x (nb*bo)
    pi = np.zeros((nb * nb, nb * nb))
    for a in range(nb):
        for c in range(nb):
            pi[a * nb + c, c * nb + a] = 1.0
    return bd1 @ pi @ bd2


def blast_dense(U: np.ndarray, V: np.ndarray, S: np.ndarray) -> np.ndarray:
    """Dense W_hat of a BLAST matrix with nb x nb blocks ([S] Appendix B: row and column bases
    shared across blocks; [B] structured-methods section: each block is a shared row basis,
    a block-specific small middle matrix and a shared column basis). U [nb, p, t]: the basis
    of block row i; V [nb, q, t]: the basis of block column j; S [nb, nb, t, t]: the middle
    matrix of block (i, j). Block (i, j) = U[i] S[i, j] V[j]^T."""
    nb, p, t = U.shape
    q = V.shape[1]
    W = np.zeros((nb * p, nb * q))
    for i in range(nb):
        for j in range(nb):
            W[i * p:(i + 1) * p, j * q:(j + 1) * q] = U[i] @ S[i, j] @ V[j].T
    return W


def blast_factors(W: np.ndarray, nb: int, t: int, sweeps: int = 10):
    """BLAST fit by minimising the reconstruction error ||W - W_hat||_F ([B] structured-methods
    section), alternating exact minimisations with orthonormal bases:
      start: U[i] = top-t left singular vectors of block row i, V[j] = top-t right singular
             vectors of block column j;
      middle matrices (bases fixed): S[i, j] = U[i]^T W_ij V[j] (the least-squares optimum);
      row bases (column bases fixed, S optimal): U[i] = top-t left singular vectors of
             [W_i1 V[1], ..., W_i,nb V[nb]] (maximises sum_j ||U[i]^T W_ij V[j]||^2);
      column bases likewise from [W_1j^T U[1], ..., W_nb,j^T U[nb]];
    `sweeps` rounds of (U, V), then S. Returns U [nb, p, t], V [nb, q, t], S [nb, nb, t, t]."""
    d, m = W.shape
    p, q = d // nb, m // nb
    if p * nb != d or q * nb != m or t > min(p, q):
        raise ValueError("BLAST needs nb | d, nb | m and t <= min(d, m) / nb")
    blk = lambda i, j: W[i * p:(i + 1) * p, j * q:(j + 1) * q]
    U = np.stack([np.linalg.svd(W[i * p:(i + 1) * p], full_matrices=False)[0][:, :t]
                  for i in range(nb)])
    V = np.stack([np.linalg.svd(W[:, j * q:(j + 1) * q], full_matrices=False)[2][:t].T
                  for j in range(nb)])
    for _ in range(sweeps):
        for i in range(nb):
            K = np.concatenate([blk(i, j) @ V[j] for j in range(nb)], axis=1)
            U[i] = np.linalg.svd(K, full_matrices=False)[0][:, :t]
        for j in range(nb):
            K = np.concatenate([blk(i, j).T @ U[i] for i in range(nb)], axis=1)
            V[j] = np.linalg.svd(K, full_matrices=False)[0][:, :t]
    S = np.stack([np.stack([U[i].T @ blk(i, j) @ V[j] for j in range(nb)]) for i in range(nb)])
    return U, V, S


def input_aware_scaling(X_cal: np.ndarray, mode: str) -> np.ndarray:
    """The input-side transform S of an input-aware decomposition, from calibration
    activations X_cal [N, d] ([S] Appendix B: input-aware methods use an activation-based
    diagonal scaling or a Cholesky factor of the input covariance; [B] structured-methods
    section: S built from calibration activations).
      "diag":     S = diag(rms of each input channel over the calibration rows);
      "cholesky": S = the lower Cholesky factor of the covariance X_cal^T X_cal / N.
    In the row-vector convention y = x W used here the output error over the calibration
    rows is ||X_cal (W - W_hat)||_F, which equals ||S^T (W - W_hat)||_F for the Cholesky
    factor (X_cal^T X_cal / N = S S^T), up to the factor sqrt(N)."""
    N = X_cal.shape[0]
    if mode == "diag":
        return np.diag(np.sqrt(np.mean(X_cal * X_cal, axis=0)))
    if mode == "cholesky":
        return np.linalg.cholesky(X_cal.T @ X_cal / N)
    raise ValueError(mode)


def input_aware_factors(W: np.ndarray, k: int, X_cal: np.ndarray, mode: str):
    """Input-aware truncated SVD ([S] Appendix B; [B] structured-methods section): write
    W = S^-T (S^T W), truncate S^T W to rank k by its SVD, and map back, so
    W_hat = S^-T TSVD_k(S^T W) (the pages' W = (W S) S^-1 with W acting on column vectors).
    Returned as U = S^-T U_k sqrt(S_k) [d x k] and V = sqrt(S_k) V_k^T [k x m]."""
    S = input_aware_scaling(X_cal, mode)
    u, sv, vt = np.linalg.svd(S.T @ W, full_matrices=False)
    root = np.sqrt(sv[:k])
    U = np.linalg.solve(S.T, u[:, :k] * root[None, :])
    return U, root[:, None] * vt[:k]


def residual(W: np.ndarray, W_hat: np.ndarray) -> np.ndarray:
    """W_res = W - W_hat. [B] residual-split section, first equation."""
    return W - W_hat


def top_right_singular(W_res: np.ndarray, r: int) -> np.ndarray:
    """R0: the top-r right singular vectors of W_res as orthonormal rows (r x m).
    [B] offline-preparation section; [S] 2.3 (for a low-rank W_hat these are W's
    singular vectors k+1..k+r)."""
    _, _, vt = np.linalg.svd(W_res, full_matrices=False)
    return vt[:r].copy()


def projection(W_res: np.ndarray, R0: np.ndarray) -> np.ndarray:
    """P = W_res R0^T (R0 R0^T)^-1: the least-squares L-update with R = R0 held fixed,
    evaluated in the pages' order (the output dimension is first reduced to r, so online
    L = X P is one thin product). [B] rank-r objective section and one-step section."""
    gram = R0 @ R0.T
    return np.linalg.solve(gram, (W_res @ R0.T).T).T


def prepare(W: np.ndarray, b: np.ndarray, kind: str, k: int, r: int,
            R0: np.ndarray | None = None, factors=None) -> dict:
    """Offline preparation [B] offline-preparation section: static fit, residual, R0, P.
    ``factors`` optionally supplies the static factors (U, V) or (B1, B2)."""
    if kind == "lowrank":
        U, V = factors if factors is not None else tsvd_factors(W, k)
        W_hat = lowrank_dense(U, V)
    elif kind == "monarch":
        U, V = factors if factors is not None else monarch_factors(W, k)
        W_hat = monarch_dense(U, V)
    elif kind == "blast":   # k = (nb, t); factors = (U, V, S)
        nb, t = k
        U, V, S = factors if factors is not None else blast_factors(W, nb, t)
        W_hat = blast_dense(U, V, S)
        prep_extra = dict(F3=S)
    else:
        raise ValueError(kind)
    W_res = residual(W, W_hat)
    if R0 is None:
        R0 = top_right_singular(W_res, r)
    P = projection(W_res, R0)
    out = dict(kind=kind, k=k, r=r, W=W, b=np.asarray(b, dtype=np.float64), F1=U, F2=V,
               W_hat=W_hat, W_res=W_res, R0=R0, P=P)
    if kind == "blast":
        out.update(prep_extra)
    return out


# ------------------------------------------------------------------------------------
# online step

def newton_schulz_inverse(G: np.ndarray, iters: int) -> np.ndarray:
    """Approximate G^-1 of an SPD matrix by Newton-Schulz ([S] 2.4: Newton-Schulz for
    larger r). Start and scaling are a reading of the pages (module docstring)."""
    dinv = 1.0 / np.sqrt(np.diag(G))
    Gh = G * dinv[:, None] * dinv[None, :]
    alpha = 1.0 / np.max(np.sum(np.abs(Gh), axis=1))
    Xt = alpha * np.eye(G.shape[0])
    two = 2.0 * np.eye(G.shape[0])
    for _ in range(iters):
        Xt = Xt @ (two - Gh @ Xt)
    return Xt * dinv[:, None] * dinv[None, :]


def solve_right_factor(G: np.ndarray, B: np.ndarray, solver: str = "cholesky",
                       ns_iters: int = 8):
    """R = G^-1 B ([B] rank-r objective section: R-update with L fixed). Returns (R, ok);
    ok is False when G is not positive definite, and then R = 0."""
    if solver == "cholesky":
        try:
            cf = sla.cho_factor(G, lower=True)
        except np.linalg.LinAlgError:
            return np.zeros_like(B), False
        if not np.all(np.isfinite(cf[0])):
            return np.zeros_like(B), False
        return sla.cho_solve(cf, B), True
    if solver == "newton_schulz":
        dg = np.diag(G)
        if not np.all(dg > 0) or not np.all(np.isfinite(G)):
            return np.zeros_like(B), False
        return newton_schulz_inverse(G, ns_iters) @ B, True
    raise ValueError(solver)


def forward(X: np.ndarray, prep: dict, ridge: float = 0.0, solver: str = "cholesky",
            ns_iters: int = 8, rows=None, keep: bool = False):
    """One-step DyRA output for X [batch, n, d].

    Per sample s ([B] one-step section, XW ~ X W_hat + L(1) R(1); [B] rank-r objective
    section for the two updates and their order of operations):
        L = X_s P                        (L-update with R0 fixed; P precomputed offline)
        G = L^T L + ridge I              ([S] 2.2: ridge for stability)
        C = L^T X_s                      (input first projected to L's r-dim space)
        B = C W_res                      (then multiplied by the residual)
        R = G^-1 B                       (Cholesky for small r, Newton-Schulz for large r, [S] 2.4)
        Y_s = X_s W_hat + b + L R
    ``rows`` (optional, one index array per sample) restricts which output rows are formed;
    L, G, C, B and R always use every token of the sample.
    Returns Y (list of arrays when rows is given), plus a dict of intermediates if keep."""
    P, W_res, W_hat, b = prep["P"], prep["W_res"], prep["W_hat"], prep["b"]
    r = P.shape[1]
    outs, inter = [], dict(L=[], G=[], C=[], B=[], R=[], ok=[])
    for s in range(X.shape[0]):
        Xs = X[s]
        L = Xs @ P
        G = L.T @ L + ridge * np.eye(r)
        C = L.T @ Xs
        B = C @ W_res
        R, ok = solve_right_factor(G, B, solver, ns_iters)
        if rows is None:
            Ys = Xs @ W_hat + b[None, :] + L @ R
        else:
            idx = np.asarray(rows[s])
            Ys = Xs[idx] @ W_hat + b[None, :] + L[idx] @ R
        outs.append(Ys)
        if keep:
            for key, val in (("L", L), ("G", G), ("C", C), ("B", B), ("R", R), ("ok", ok)):
                inter[key].append(val)
    Y = outs if rows is not None else (np.stack(outs) if outs else np.zeros((0,) + X.shape[1:2] + (W_hat.shape[1],)))
    return (Y, inter) if keep else Y


def als_factors(Xs: np.ndarray, W_res: np.ndarray, R0: np.ndarray, t: float,
                ridge: float = 0.0):
    """ALS on min ||X W_res - L R||_F^2 from R = R0 ([B] rank-r objective section;
    [S] 3.3 / Figure 9: t = 1 is L then R, t = 1.5 is L, R, L, t = 2 is L, R, L, R).
    L-update: L = X (W_res R^T (R R^T)^-1) -- output dimension reduced first.
    R-update: R = (L^T L + ridge I)^-1 (L^T X) W_res -- input projected first."""
    half_steps = int(round(2 * t))
    R = R0
    L = None
    r = R0.shape[0]
    for step in range(half_steps):
        if step % 2 == 0:
            L = Xs @ projection(W_res, R)
        else:
            G = L.T @ L + ridge * np.eye(r)
            R = np.linalg.solve(G, (L.T @ Xs) @ W_res)
    return L, R


def forward_als(X: np.ndarray, prep: dict, t: float, ridge: float = 0.0,
                solver: str = "cholesky", ns_iters: int = 8):
    """DyRA output with t ALS iterations ([S] 3.3 / Figure 9; [B] ablation paragraph: t = 1,
    1.5, 2, where 1.5 updates L, R, L), per sample, in the rank-r objective's order of
    operations ([B] rank-r objective section):
        L-update (R fixed): P = W_res R^T (R R^T)^-1, L = X P   (the first one from R0 is
                            the offline P)
        R-update (L fixed): R = (L^T L + ridge I)^-1 (L^T X) W_res
    alternating for round(2 t) half-steps from R0, then Y_s = X_s W_hat + b + L R. Both
    solves use `solver` (Cholesky, or the Newton-Schulz mirror). t = 1 is forward()."""
    W_hat, W_res, b, R0, P0 = prep["W_hat"], prep["W_res"], prep["b"], prep["R0"], prep["P"]
    r = R0.shape[0]
    outs = []
    for s in range(X.shape[0]):
        Xs = X[s]
        R, L = R0, None
        for step in range(int(round(2 * t))):
            if step == 0:
                L = Xs @ P0
            elif step % 2 == 0:
                Pt, _ = solve_right_factor(R @ R.T, R @ W_res.T, solver, ns_iters)   # P^T
                L = Xs @ Pt.T
            else:
                G = L.T @ L + ridge * np.eye(r)
                R, _ = solve_right_factor(G, (L.T @ Xs) @ W_res, solver, ns_iters)
        outs.append(Xs @ W_hat + b[None, :] + L @ R)
    return np.stack(outs)


def gelu(x: np.ndarray) -> np.ndarray:
    """GELU(x) = x Phi(x) = x (1 + erf(x / sqrt 2)) / 2, the erf form used by the ViT and DINOv3
    MLP blocks the pages evaluate ([S] Appendix D, their MLP layers)."""
    from scipy.special import erf
    return 0.5 * x * (1.0 + erf(x / np.sqrt(2.0)))


def mlp_forward(X: np.ndarray, prep1: dict, prep2: dict, ridge: float = 0.0,
                solver: str = "cholesky", ns_iters: int = 8):
    """A transformer MLP block with both linear layers replaced by DyRA ([S] Appendix D: every
    linear layer of the evaluated models is replaced): H = GELU(DyRA_fc1(X)), then
    Y = DyRA_fc2(H), each layer's correction computed from its own input."""
    H = gelu(forward(X, prep1, ridge=ridge, solver=solver, ns_iters=ns_iters))
    return forward(H, prep2, ridge=ridge, solver=solver, ns_iters=ns_iters)


# ------------------------------------------------------------------------------------
# metrics

def relative_frobenius(a: np.ndarray, b: np.ndarray) -> float:
    den = float(np.linalg.norm(b))
    return float(np.linalg.norm(a - b)) / (den if den > 0 else 1.0)


def approximation_error(Y: np.ndarray, X: np.ndarray, W: np.ndarray, b: np.ndarray) -> float:
    """E = ||Y - b - X W||_F / ||X W||_F over the whole batch (the quantity the paper's
    output-error figures report, [S] 2.3 / Figure 3 and E.4)."""
    XW = X @ W
    return float(np.linalg.norm(Y - b - XW)) / float(np.linalg.norm(XW))
