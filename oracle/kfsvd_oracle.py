"""fp64 CPU oracle for curvature-whitened truncated SVD with global rank allocation.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or execute
this module: only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` use it.  It shares no code with the CUDA library; the only thing both sides
use is the seeded input generator in ``synth`` (which holds no method arithmetic).

Every function is a plain, slow, directly checkable statement of what the pages define,
in float64 (numpy/LAPACK routines serve as textbook steps).  Sources:

  [LASER]   "LASER: Loss-Aware Singular-value Decomposition and Rank Allocation for
            Efficient Low-Precision Vision-Language Models", technical summary,
            Methodology 1 (K-FAC surrogate, curvature-weighted transformation,
            quantisation-aware whitening) and 2 (global greedy rank allocation).
  [UniRank] "UniRank: Unified Rank Allocation for Low-Rank LLM Compression",
            section 2.1 (sort all scores descending, accumulate the m+n cost of each kept
            singular pair until the parameter budget is reached).
  [Swift]   "Swift-SVD: Theoretical Optimality Meets Practical Efficiency in Low-Rank LLM
            Compression", section 2A (closed form W_k = W V_k V_k^T; incremental
            covariance aggregation; one eigendecomposition of the aggregated covariance)
            and section B (hybrid scoring of layer importance and closed-form loss for the
            dynamic rank allocation).

Readings where the pages are silent: W is d_in x d_out (y = x W);
X = A^T A / N and G = Gr^T Gr / N uncentred, each damped by lam * mean(diag); the
Cholesky factors are S_x = chol_lower(X)^T and S_g = chol_lower(G), which is the choice
that makes ||S_x dW S_g||_F^2 equal the K-FAC form with column-major vec; the score of a
component is half its squared whitened singular value; the greedy cut keeps the longest
prefix of the sorted list whose cumulative cost stays within the budget; an attention head
is a unit of its own (LASER 2 allocates across heads): q, k and v heads are column blocks of
their weight with the head's diagonal block of G, o heads are row blocks with the head's
diagonal block of X, each block taken from the factor after damping.

Parity status: every function here is pinned by tests/test_oracle_pins.py against
closed forms, the pages' identities, brute force or hand-worked values; none is
"parity unpinned".
"""
from __future__ import annotations

import math
from dataclasses import dataclass
from typing import Dict, List, Optional, Sequence

import numpy as np
import scipy.linalg as sla

KEY_HALF_SIGMA2 = "half_sigma2"
KEY_PER_PARAM = "per_param"
KEY_ENERGY_RATIO = "energy_ratio"
FIXED_RANK = "fixed_rank"


# --------------------------------------------------------------- step 1: covariances
def covariance_sum(A: np.ndarray) -> np.ndarray:
    """Running second-moment sum A^T A of a block of calibration rows (tokens x channels).

    [Swift] 2A, incremental aggregation: the covariance is a sum over tokens of outer
    products, so it can be accumulated batch by batch.
    """
    A = np.asarray(A, dtype=np.float64)
    return A.T @ A


def finalize_covariance(S: np.ndarray, n_tokens: int, lam: float) -> np.ndarray:
    """X = S / N, then X + lam * mean(diag(X)) * I.  [LASER] 1: covariance over the
    calibration set; normalisation and damping follow the statement of the hot path."""
    C = np.asarray(S, dtype=np.float64) / float(n_tokens)
    return C + lam * np.mean(np.diag(C)) * np.eye(C.shape[0])


def fake_quant_int8_token(A: np.ndarray) -> np.ndarray:
    """Quantisation-aware whitening input: per-token symmetric INT8 fake quantisation.

    [LASER] 1 (QAW): the K-FAC factors are estimated from quantised calibration
    activations.  The page gives no quantiser; this is the plain symmetric per-row one:
    scale s_t = max_j |A_tj| / 127, code q = clamp(rint(A_tj / s_t), -127, 127) with
    round-half-even, output s_t * q rounded to bfloat16 (a zero row stays zero).  The
    scale and the code decide integers, so this step runs in float32 exactly as the
    kernel does (IEEE division and multiplication), not in float64.
    """
    A = np.asarray(A, dtype=np.float32)
    amax = np.max(np.abs(A), axis=1, keepdims=True).astype(np.float32)
    s = (amax / np.float32(127.0)).astype(np.float32)
    safe = np.where(s > 0, s, np.float32(1.0)).astype(np.float32)
    q = np.clip(np.rint((A / safe).astype(np.float32)), -127, 127).astype(np.float32)
    y = (s * q).astype(np.float32)
    y = np.where(s > 0, y, np.float32(0.0)).astype(np.float32)
    u = y.view(np.uint32)
    with np.errstate(over="ignore"):
        r = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return (r.astype(np.uint32) << np.uint32(16)).view(np.float32)


# -------------------------------------------------------------- step 2: factors
def cholesky_factors(X: np.ndarray, G: np.ndarray):
    """S_x = chol_lower(X)^T (upper), S_g = chol_lower(G) (lower).  [LASER] 1: S_x, S_g
    are Cholesky factors of X and G; this orientation gives S_x^T S_x = X, S_g S_g^T = G."""
    Lx = sla.cholesky(np.asarray(X, dtype=np.float64), lower=True, check_finite=False)
    Lg = sla.cholesky(np.asarray(G, dtype=np.float64), lower=True, check_finite=False)
    return Lx.T.copy(), Lg


# --------------------------------------------------------------- step 3: whitening
def whiten(W: np.ndarray, Sx: np.ndarray, Sg: np.ndarray) -> np.ndarray:
    """[LASER] 1: curvature-weighted weight W~ = S_x W S_g."""
    return Sx @ np.asarray(W, dtype=np.float64) @ Sg


# ------------------------------------------------------------- step 4: spectrum
def whitened_svd(Wt: np.ndarray):
    """[LASER] 1: SVD of W~ (LAPACK gesdd).  Returns (U~, sigma descending, V~)."""
    U, s, Vt = np.linalg.svd(Wt, full_matrices=False)
    return U, s, Vt.T


def gram_eigenvalues(Wt: np.ndarray) -> np.ndarray:
    """[Swift] 2A: one eigendecomposition of the Gram matrix of the smaller side."""
    m, n = Wt.shape
    C = Wt.T @ Wt if n <= m else Wt @ Wt.T
    w = np.linalg.eigvalsh(C)   # the eigenvalues alone: the spectrum is all this step returns
    return np.sort(w)[::-1]


# ----------------------------------------------------------- step 5: allocation
def component_scores(sigma: np.ndarray, cost: int, mode: str, precision: str, weight: Optional[float] = None):
    """Score of each component: half its squared whitened singular value (the K-FAC
    estimate of the loss increase when it is dropped, [LASER] 1), or that divided by the
    m+n parameters the pair costs ([LASER] 2, "score per parameter cost"), or [UniRank] 2.1's
    local structural significance, the energy ratio sigma_i^2 / ||Sigma||_F^2 of the unit.
    A unit weight (UniRank's functional importance I_l) multiplies every key of the unit;
    a weight that is not positive gives 0.

    ``precision="f32"`` evaluates the key in float32 with one rounding per operation, the
    order the GPU uses (square, divide, multiply by the weight; the energy is the float64 sum
    of the squares rounded to float32), so that both sides rank identical float32 sigma
    identically.
    """
    if precision == "f32":
        s = np.asarray(sigma, dtype=np.float32)
        q = (s * s).astype(np.float32)
        if mode == KEY_ENERGY_RATIO:
            e = np.float32(np.sum(np.asarray(s, dtype=np.float64) ** 2))
            sc = (q / e).astype(np.float32) if e > 0 else np.zeros_like(q)
        else:
            sc = (np.float32(0.5) * q).astype(np.float32)
            if mode == KEY_PER_PARAM:
                sc = (sc / np.float32(cost)).astype(np.float32)
        if weight is not None:
            w = np.float32(weight)
            sc = (w * sc).astype(np.float32) if w > 0 else np.zeros_like(sc)
        return sc
    s = np.asarray(sigma, dtype=np.float64)
    if mode == KEY_ENERGY_RATIO:
        e = float(np.sum(s * s))
        sc = s * s / e if e > 0 else np.zeros_like(s)
    else:
        sc = 0.5 * s * s
        if mode == KEY_PER_PARAM:
            sc = sc / float(cost)
    if weight is not None:
        sc = sc * float(weight) if weight > 0 else np.zeros_like(sc)
    return sc


@dataclass
class Allocation:
    ranks: np.ndarray          # int64 per unit
    cut_score: float           # score of the last kept component (nan if none kept)
    next_score: float          # score of the first dropped component (nan if none)
    used: int                  # parameters used by the kept components
    order_unit: np.ndarray     # sorted list: unit of each component
    order_comp: np.ndarray     # sorted list: index of each component inside its unit
    order_score: np.ndarray


def allocate(sigmas: Sequence[np.ndarray], costs: Sequence[int], budget: int,
             mode: str = KEY_HALF_SIGMA2, fixed_ranks: Optional[Sequence[int]] = None,
             precision: str = "f64", weights: Optional[Sequence[float]] = None) -> Allocation:
    """Global sort-and-truncate rank allocation.

    [UniRank] 2.1 and [LASER] 2: pool the scores of every component of every unit, sort
    them descending (ties: lower unit index first, then lower component index), walk the
    list accumulating each component's parameter cost m+n, and keep the longest prefix
    whose cumulative cost does not exceed the budget.  The rank of a unit is the number
    of its components in that prefix.
    """
    n_units = len(sigmas)
    if mode == FIXED_RANK:
        ranks = np.array([min(int(fixed_ranks[u]), len(sigmas[u])) for u in range(n_units)])
        used = int(sum(int(ranks[u]) * int(costs[u]) for u in range(n_units)))
        e = np.zeros(0, dtype=np.int64)
        return Allocation(ranks, float("nan"), float("nan"), used, e, e, np.zeros(0))
    units, comps, scores = [], [], []
    for u, s in enumerate(sigmas):
        sc = component_scores(s, costs[u], mode, precision, None if weights is None else weights[u])
        units.append(np.full(len(sc), u, dtype=np.int64))
        comps.append(np.arange(len(sc), dtype=np.int64))
        scores.append(sc.astype(np.float64))
    units = np.concatenate(units)
    comps = np.concatenate(comps)
    scores = np.concatenate(scores)
    order = np.lexsort((comps, units, -scores))
    cost_sorted = np.asarray(costs, dtype=np.int64)[units[order]]
    prefix = np.cumsum(cost_sorted)
    n_keep = int(np.searchsorted(prefix, budget, side="right"))
    ranks = np.bincount(units[order[:n_keep]], minlength=n_units).astype(np.int64)
    cut = float(scores[order[n_keep - 1]]) if n_keep > 0 else float("nan")
    nxt = float(scores[order[n_keep]]) if n_keep < len(order) else float("nan")
    used = int(prefix[n_keep - 1]) if n_keep > 0 else 0
    return Allocation(ranks, cut, nxt, used, units[order], comps[order], scores[order])


# --------------------------------------------------------- step 5: map back
def unwhiten(Sx: np.ndarray, Sg: np.ndarray, Ut: np.ndarray, sigma: np.ndarray,
             Vt: np.ndarray, r: int):
    """[LASER] 1: map the rank-r factors of W~ back to the original space:
    U = S_x^-1 U~_r Sigma_r (d_in x r) and V = V~_r^T S_g^-1 (r x d_out), by triangular
    solves (S_x upper, S_g lower)."""
    B = Ut[:, :r] * sigma[:r][None, :]
    U = sla.solve_triangular(Sx, B, lower=False)
    V = sla.solve_triangular(Sg.T, Vt[:, :r], lower=False).T
    return U, V


# ------------------------------------------------ empirical-Fisher component scores
def empirical_fisher_scores(A: np.ndarray, Gr: np.ndarray, U: np.ndarray, V: np.ndarray) -> np.ndarray:
    """[LASER] 2: the importance of component i is its contribution to the empirical-Fisher
    quadratic loss, evaluated with the calibration gradients in the original space:
    score_i = 1/2 (1/N) sum_t (a_t . u_i)^2 (g_t . v_i)^2, with u_i the i-th column of U
    (d_in x r) and v_i the i-th row of V (r x d_out).  This is 1/2 vec(dW)^T F vec(dW) for the
    rank-one dW = u_i v_i and F = (1/N) sum_t vec(a_t^T g_t) vec(a_t^T g_t)^T."""
    A = np.asarray(A, dtype=np.float64)
    Gr = np.asarray(Gr, dtype=np.float64)
    P = A @ np.asarray(U, dtype=np.float64)            # N x r: a_t . u_i
    Q = Gr @ np.asarray(V, dtype=np.float64).T         # N x r: g_t . v_i
    return 0.5 * np.mean(P * P * Q * Q, axis=0)


def allocate_keys(keys: Sequence[np.ndarray], costs: Sequence[int], budget: int) -> Allocation:
    """Sort-and-truncate over arbitrary non-negative per-component keys ([UniRank] 2.1's
    procedure with any score, e.g. [LASER] 2's empirical-Fisher scores, which are not
    monotone along a unit's spectrum): ties by unit, then component index; the kept set of a
    unit is then any subset, returned as order_unit/order_comp of the first `ranks.sum()`
    entries and by the per-unit counts."""
    units, comps, scores = [], [], []
    for u, k in enumerate(keys):
        k = np.asarray(k, dtype=np.float64)
        units.append(np.full(len(k), u, dtype=np.int64))
        comps.append(np.arange(len(k), dtype=np.int64))
        scores.append(k)
    units = np.concatenate(units)
    comps = np.concatenate(comps)
    scores = np.concatenate(scores)
    order = np.lexsort((comps, units, -scores))
    prefix = np.cumsum(np.asarray(costs, dtype=np.int64)[units[order]])
    n_keep = int(np.searchsorted(prefix, budget, side="right"))
    ranks = np.bincount(units[order[:n_keep]], minlength=len(keys)).astype(np.int64)
    cut = float(scores[order[n_keep - 1]]) if n_keep > 0 else float("nan")
    nxt = float(scores[order[n_keep]]) if n_keep < len(order) else float("nan")
    used = int(prefix[n_keep - 1]) if n_keep > 0 else 0
    return Allocation(ranks, cut, nxt, used, units[order], comps[order], scores[order])


def swift_residual_losses(sigma: np.ndarray) -> List[float]:
    """[Swift] 2A/B: the closed-form loss of a unit truncated to rank k is the energy of the
    components it drops, eps*_k = sum_{j >= k} sigma_j^2 (k = 0 .. len - 1, 0-based sigma).
    Summed in float64 from the last component upward, one term at a time (the square of a
    float32 value is exact in float64), so that the sum order is fixed."""
    s = [float(np.float32(x)) for x in sigma]
    eps = [0.0] * len(s)
    acc = 0.0
    for j in range(len(s) - 1, -1, -1):
        acc = acc + s[j] * s[j]
        eps[j] = acc
    return eps


def swift_hybrid_keys(sigma: np.ndarray, beta: float, alpha: float) -> np.ndarray:
    """[Swift] B, hybrid scoring s_i = beta_i^alpha (log(e + eps*_{k,i}))^(1 - alpha) as a
    sort-and-truncate key per component: component k (0-based) of unit i gets the unit's
    score at rank k, i.e. while it holds the k components before it, so the next component
    always goes to the unit whose current truncation scores highest (keys sorted
    descending).  eps*_k is non-increasing in k, so every unit's keys are too and the kept
    set is a prefix of its spectrum.  beta_i (the unit's end-to-end importance) and alpha in
    [0, 1] are the caller's; a beta that is not positive gives the unit keys 0.  Each key is
    evaluated in float64 with the C library's log and pow and rounded once to float32."""
    eps = swift_residual_losses(sigma)
    b = float(np.float32(beta))      # the importance is given as a float32 per unit
    if not (b > 0.0):
        return np.zeros(len(eps), dtype=np.float32)
    bw = math.pow(b, float(alpha))
    out = np.empty(len(eps), dtype=np.float32)
    for k, e in enumerate(eps):
        out[k] = np.float32(bw * math.pow(math.log(math.e + e), 1.0 - float(alpha)))
    return out


def allocate_swift_hybrid(sigmas: Sequence[np.ndarray], costs: Sequence[int], budget: int,
                          betas: Sequence[float], alpha: float) -> Allocation:
    """Global sort-and-truncate ([UniRank] 2.1's procedure) on [Swift] B's hybrid keys."""
    return allocate_keys([swift_hybrid_keys(s, b, alpha) for s, b in zip(sigmas, betas)], costs, budget)


def hybrid_ffn_budget(budget: int, d_model: Sequence[int], n_dense: Sequence[int]) -> int:
    """[LASER] hybrid FFN: the parameter budget left for the low-rank factors once the dense
    channels are paid for, max(budget - sum_p d_model_p n_dense_p, 0); each dense channel of a
    gate or up projection keeps its d_model weights (one entry per projection)."""
    left = int(budget) - sum(int(a) * int(b) for a, b in zip(d_model, n_dense))
    return max(left, 0)


# --------------------------------------------------------------- the objective
def kfac_quadratic(dW: np.ndarray, X: np.ndarray, G: np.ndarray) -> float:
    """[LASER] 1, K-FAC surrogate: 1/2 vec(dW)^T (G kron X) vec(dW), built explicitly
    (tiny shapes only), vec stacking the columns of dW (d_in x d_out)."""
    v = np.asarray(dW, dtype=np.float64).reshape(-1, order="F")
    K = np.kron(np.asarray(G, dtype=np.float64), np.asarray(X, dtype=np.float64))
    return 0.5 * float(v @ K @ v)


def whitened_error(W: np.ndarray, U: np.ndarray, V: np.ndarray, Sx: np.ndarray,
                   Sg: np.ndarray) -> float:
    """||S_x (W - U V) S_g||_F^2, twice the K-FAC loss estimate of replacing W by U V."""
    D = Sx @ (np.asarray(W, dtype=np.float64) - np.asarray(U, np.float64) @ np.asarray(V, np.float64)) @ Sg
    return float(np.sum(D * D))


# ------------------------------------------------ Swift-SVD activation-only route
def output_covariance(A: np.ndarray, W: np.ndarray) -> np.ndarray:
    """[Swift] 2A: the covariance of the layer output aggregated over the calibration tokens,
    C = (1/N) sum_t y_t^T y_t with y_t = a_t W (row t of Y = A W)."""
    Y = np.asarray(A, dtype=np.float64) @ np.asarray(W, dtype=np.float64)
    return Y.T @ Y / A.shape[0]


def output_eig(C: np.ndarray):
    """[Swift] 2A: one eigendecomposition of C.  Returns sigma = sqrt(max(lambda, 0)) in
    descending order (the singular values of Y / sqrt(N)) and the eigenvectors as columns."""
    lam, V = np.linalg.eigh(np.asarray(C, dtype=np.float64))
    order = np.argsort(-lam, kind="stable")
    return np.sqrt(np.maximum(lam[order], 0.0)), V[:, order]


def activation_factors(W: np.ndarray, V: np.ndarray, k: int):
    """[Swift] 2A closed form W_k = W V_k V_k^T, as the factors U = W V_k (d_in x k) and
    V_k^T (k x d_out)."""
    Vk = np.asarray(V, dtype=np.float64)[:, :k]
    return np.asarray(W, dtype=np.float64) @ Vk, Vk.T.copy()


def activation_loss(A: np.ndarray, W: np.ndarray, U: np.ndarray, V: np.ndarray) -> float:
    """(1/N) ||A W - A U V||_F^2: the activation-aware reconstruction loss [Swift] 2A
    minimises."""
    A = np.asarray(A, dtype=np.float64)
    D = A @ (np.asarray(W, np.float64) - np.asarray(U, np.float64) @ np.asarray(V, np.float64))
    return float(np.sum(D * D)) / A.shape[0]


def compress_workload_activation_only(wl, units: Optional[List[int]] = None, chunk: int = 8192) -> Dict:
    """The activation-only route on a synthetic workload: per unit the output covariance of
    its calibration rows (fake-quantised first under quantisation-aware whitening; a head
    unit reads its block of the input channels), one eigendecomposition, the global
    sort-and-truncate on 1/2 sigma^2 over the first min(m, n) components of every unit
    (rank(Y) <= min(m, n)), and the factors W V_k, V_k^T."""
    from synth import recipes
    idx = list(range(len(wl.units))) if units is None else list(units)
    out = []
    for i in idx:
        u = wl.units[i]
        site = wl.sites[u.x_site]
        W = recipes.gen_weight(wl, u).astype(np.float64)
        C = np.zeros((u.n, u.n))
        for t0 in range(0, wl.n_tokens, chunk):
            A = recipes.gen_stream(wl, site, t0, min(wl.n_tokens, t0 + chunk))
            if wl.quant == "int8_token":
                A = fake_quant_int8_token(A)
            C += output_covariance(A[:, u.x_off:u.x_off + u.m], W) * A.shape[0]
        C /= wl.n_tokens
        sig, V = output_eig(C)
        out.append({"name": u.name, "m": u.m, "n": u.n, "C": C, "sigma": sig, "V": V, "W": W})
    sigs = [o["sigma"][:min(o["m"], o["n"])] for o in out]
    alloc = allocate(sigs, [o["m"] + o["n"] for o in out], wl.budget)
    for o, k in zip(out, alloc.ranks):
        o["rank"] = int(k)
        o["U"], o["Vt"] = activation_factors(o["W"], o["V"], int(k))
    return {"units": out, "alloc": alloc}


# ------------------------------------------------ LASER hybrid FFN channel selection
def channel_errors(W: np.ndarray, U: np.ndarray, V: np.ndarray, X: np.ndarray) -> np.ndarray:
    """[LASER] hybrid FFN: the reconstruction error of every hidden channel j (column j of a
    gate or up projection, d_model x d_ffn) under a temporary low-rank approximation U V:
    e_j = d_j^T X d_j with d_j = (W - U V)[:, j], i.e. the mean squared error of channel j's
    pre-activation over the calibration inputs when X = A^T A / N."""
    D = np.asarray(W, np.float64) - np.asarray(U, np.float64) @ np.asarray(V, np.float64)
    return np.einsum("ij,ik,kj->j", D, np.asarray(X, np.float64), D)


def select_svd_channels(errors: Sequence[np.ndarray], n_svd: int) -> np.ndarray:
    """[LASER] hybrid FFN: the n_svd "SVD-friendly" hidden channels, those with the lowest
    summed reconstruction error over the projections that share the channel (gate and up).
    Stated the other way round: the len - n_svd channels with the largest error stay dense,
    ties to the lower channel index.  Returned in increasing channel order."""
    e = np.sum([np.asarray(x, np.float64) for x in errors], axis=0)
    order = np.lexsort((np.arange(len(e)), -e))
    return np.sort(order[len(e) - n_svd:])


def compress_hybrid_ffn(wl, r_temp: int, n_svd: int, pairs=None) -> Dict:
    """[LASER] hybrid FFN over a workload: every other unit as in compress_workload; for each
    (gate, up) pair, the temporary whitened SVD at rank r_temp scores the hidden channels
    (channel_errors, summed over gate and up), the n_svd lowest-error channels form the
    SVD-friendly set S and the rest stay dense.  The SVD branch is gate[:, S] and up[:, S],
    each whitened with its unit's X and the block G[S, S] of its gradient factor and entered
    into the global allocation; the dense channels cost d_model parameters each, per
    projection, taken off the budget first.  ``pairs``: (gate, up) unit-index pairs (default:
    the units named gate and up of each block)."""
    from synth import recipes
    if pairs is None:
        pairs = []
        for b in sorted({u.block for u in wl.units}):
            idx = {u.name.split(".")[-1]: i for i, u in enumerate(wl.units) if u.block == b}
            pairs.append((idx["gate"], idx["up"]))
    ref = compress_workload(wl)
    covs = ref["covs"]
    units = ref["units"]
    in_pair = {i for p in pairs for i in p}
    entries = []          # (kind, unit index, UnitResult-like dict)
    for i, ur in enumerate(units):
        if i not in in_pair:
            entries.append(("unit", i, ur))
    splits = []
    dense_cost = 0
    for gi, ui in pairs:
        errs = []
        for i in (gi, ui):
            ur = units[i]
            U, V = unwhiten(ur.Sx, ur.Sg, ur.U_t, ur.sigma, ur.V_t, r_temp)
            errs.append(channel_errors(recipes.gen_weight(wl, wl.units[i]), U, V, ur.X))
        S = select_svd_channels(errs, n_svd)
        f = units[gi].n
        D = np.setdiff1d(np.arange(f), S)
        splits.append({"gate": gi, "up": ui, "svd": S, "dense": D, "errors": errs[0] + errs[1]})
        for i in (gi, ui):
            ur = units[i]
            dense_cost += ur.m * len(D)
            if len(S) == 0:
                continue
            W = recipes.gen_weight(wl, wl.units[i]).astype(np.float64)[:, S]
            G = ur.G[np.ix_(S, S)]
            Sx, Sg = cholesky_factors(ur.X, G)
            Wt = whiten(W, Sx, Sg)
            Ut, sg, Vt = whitened_svd(Wt)
            entries.append(("svd", i, UnitResult(ur.name + ".svd", ur.m, len(S), ur.X, G, Sx, Sg, Wt, Ut, sg, Vt)))
    costs = [e[2].m + e[2].n for e in entries]
    budget = wl.budget - dense_cost
    alloc = allocate([e[2].sigma for e in entries], costs, max(budget, 0))
    for e, k in zip(entries, alloc.ranks):
        r = e[2]
        r.rank = int(k)
        r.U, r.V = unwhiten(r.Sx, r.Sg, r.U_t, r.sigma, r.V_t, r.rank)
    return {"entries": entries, "splits": splits, "alloc": alloc, "budget": budget, "dense_cost": dense_cost,
            "covs": covs}


# ------------------------------------------------------------ whole workloads
@dataclass
class UnitResult:
    name: str
    m: int
    n: int
    X: np.ndarray
    G: np.ndarray
    Sx: np.ndarray
    Sg: np.ndarray
    Wt: np.ndarray
    U_t: np.ndarray
    sigma: np.ndarray
    V_t: np.ndarray
    rank: int = 0
    U: Optional[np.ndarray] = None
    V: Optional[np.ndarray] = None


def site_covariance_sum(wl, site, chunk: int = 8192) -> np.ndarray:
    """Sum of A^T A over all calibration tokens of one site, streamed in token chunks."""
    from synth import recipes
    S = np.zeros((site.d, site.d), dtype=np.float64)
    for t0 in range(0, wl.n_tokens, chunk):
        A = recipes.gen_stream(wl, site, t0, min(wl.n_tokens, t0 + chunk))
        if wl.quant == "int8_token" and site.kind == "act":
            A = fake_quant_int8_token(A)
        S += covariance_sum(A)
    return S


def compress_workload(wl, units: Optional[List[int]] = None) -> Dict:
    """Runs the whole path on a synthetic workload: covariances of every site, factors,
    whitening and SVD of every unit, global allocation (or fixed rank), factors U, V."""
    from synth import recipes
    idx = list(range(len(wl.units))) if units is None else list(units)
    covs: Dict[str, np.ndarray] = {}

    def cov(name):
        if name not in covs:
            covs[name] = finalize_covariance(site_covariance_sum(wl, wl.sites[name]),
                                             wl.n_tokens, wl.lam)
        return covs[name]

    res: List[UnitResult] = []
    for i in idx:
        u = wl.units[i]
        # an attention-head unit uses the diagonal blocks of its (already damped) factors
        X = cov(u.x_site)[u.x_off:u.x_off + u.m, u.x_off:u.x_off + u.m]
        G = cov(u.g_site)[u.g_off:u.g_off + u.n, u.g_off:u.g_off + u.n]
        Sx, Sg = cholesky_factors(X, G)
        W = recipes.gen_weight(wl, u).astype(np.float64)
        Wt = whiten(W, Sx, Sg)
        Ut, s, Vt = whitened_svd(Wt)
        res.append(UnitResult(u.name, u.m, u.n, X, G, Sx, Sg, Wt, Ut, s, Vt))
    costs = [r.m + r.n for r in res]
    if wl.fixed_rank is not None:
        alloc = allocate([r.sigma for r in res], costs, 0, FIXED_RANK,
                         [wl.fixed_rank] * len(res))
    else:
        alloc = allocate([r.sigma for r in res], costs, wl.budget)
    for r, k in zip(res, alloc.ranks):
        r.rank = int(k)
        r.U, r.V = unwhiten(r.Sx, r.Sg, r.U_t, r.sigma, r.V_t, r.rank)
    return {"units": res, "alloc": alloc, "covs": covs}
