"""Pins of the fp64 oracle against what the pages and the mathematics fix (CPU only).

Each test is chosen so that a plausible slip in the oracle (a dropped term, a transposed
factor, the wrong vec order, a wrong damping or normalisation, a wrong cut rule) fails.
"""
import itertools
import json
import os

import numpy as np
import pytest

import oracle as O

GOLD = os.path.join(os.path.dirname(__file__), "golden")
rng = np.random.default_rng(20260602)


def _tiny_problem(m=5, n=7, N=50, lam=1e-2, seed=0):
    r = np.random.default_rng(seed)
    A = r.standard_normal((N, m)) * (1.0 / np.sqrt(np.arange(1, m + 1)))
    Gr = r.standard_normal((N, n)) * 1e-3
    W = r.standard_normal((m, n)) * 0.02
    X = O.finalize_covariance(O.covariance_sum(A), N, lam)
    G = O.finalize_covariance(O.covariance_sum(Gr), N, lam)
    return A, Gr, W, X, G


def test_covariance_hand_values():
    g = json.load(open(os.path.join(GOLD, "cov_hand.json")))
    A = np.array(g["A"], dtype=np.float64)
    np.testing.assert_array_equal(O.covariance_sum(A), np.array(g["sum"]))
    np.testing.assert_allclose(O.finalize_covariance(O.covariance_sum(A), A.shape[0], g["lam"]),
                               np.array(g["X"]), rtol=0, atol=1e-14)


def test_covariance_is_streamable():
    """Swift-SVD 2A: aggregating batch by batch equals one pass over all tokens."""
    A = rng.standard_normal((97, 6))
    S = O.covariance_sum(A[:40]) + O.covariance_sum(A[40:71]) + O.covariance_sum(A[71:])
    brute = np.zeros((6, 6))
    for t in range(A.shape[0]):
        brute += np.outer(A[t], A[t])
    np.testing.assert_allclose(S, brute, rtol=1e-13)


def test_cholesky_reconstruction_and_orientation():
    _, _, _, X, G = _tiny_problem(m=9, n=11)
    Sx, Sg = O.cholesky_factors(X, G)
    assert np.allclose(np.tril(Sx, -1), 0) and np.all(np.diag(Sx) > 0)   # upper
    assert np.allclose(np.triu(Sg, 1), 0) and np.all(np.diag(Sg) > 0)    # lower
    assert np.linalg.norm(Sx.T @ Sx - X) / np.linalg.norm(X) <= 1e-13
    assert np.linalg.norm(Sg @ Sg.T - G) / np.linalg.norm(G) <= 1e-13


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_kronecker_identity(seed):
    """LASER 1: 1/2 vec(dW)^T (G kron X) vec(dW) (explicit Kronecker, column-major vec)
    equals 1/2 ||S_x dW S_g||_F^2 for the oracle's factors and whitening."""
    _, _, W, X, G = _tiny_problem(seed=seed)
    Sx, Sg = O.cholesky_factors(X, G)
    for dW in (rng.standard_normal(W.shape), W):
        lhs = O.kfac_quadratic(dW, X, G)
        rhs = 0.5 * np.sum(O.whiten(dW, Sx, Sg) ** 2)
        assert abs(lhs - rhs) <= 1e-12 * abs(lhs)


@pytest.mark.parametrize("r", [0, 1, 3, 5])
def test_truncation_loss_equals_discarded_spectrum(r):
    """The K-FAC loss of W - U V equals half the sum of the discarded sigma^2 (LASER 1:
    truncating the smallest components gives the smallest estimated loss increase), and
    Swift-SVD's stability claim: the achieved loss is the theoretical minimum."""
    _, _, W, X, G = _tiny_problem(seed=7)
    Sx, Sg = O.cholesky_factors(X, G)
    Ut, s, Vt = O.whitened_svd(O.whiten(W, Sx, Sg))
    U, V = O.unwhiten(Sx, Sg, Ut, s, Vt, r)
    assert U.shape == (W.shape[0], r) and V.shape == (r, W.shape[1])
    dl = O.kfac_quadratic(W - U @ V, X, G)
    scale = 0.5 * np.sum(s ** 2)          # full energy: the reference size for rounding
    assert abs(dl - 0.5 * np.sum(s[r:] ** 2)) <= 1e-10 * scale
    assert abs(O.whitened_error(W, U, V, Sx, Sg) - 2 * dl) <= 1e-10 * scale


def test_eckart_young_beats_random_factorisations():
    _, _, W, X, G = _tiny_problem(m=6, n=8, seed=3)
    Sx, Sg = O.cholesky_factors(X, G)
    Ut, s, Vt = O.whitened_svd(O.whiten(W, Sx, Sg))
    for r in (1, 2, 4):
        U, V = O.unwhiten(Sx, Sg, Ut, s, Vt, r)
        e_opt = O.whitened_error(W, U, V, Sx, Sg)
        for k in range(1000):
            if k % 2 == 0:
                P, Q = rng.standard_normal((6, r)) * 0.03, rng.standard_normal((r, 8))
            else:
                eps = 10.0 ** rng.uniform(-6, -1)
                P = U + eps * rng.standard_normal(U.shape) * np.abs(U).max()
                Q = V + eps * rng.standard_normal(V.shape) * np.abs(V).max()
            assert O.whitened_error(W, P, Q, Sx, Sg) >= e_opt * (1 - 1e-12)


def test_swift_svd_closed_form_special_case():
    """Swift-SVD 2A: with G = I and no damping, the optimum of ||A W - A W_k|| is
    W_k = W V_k V_k^T with V_k the top right singular vectors of Y = A W, and the
    whitened spectrum is the spectrum of A W / sqrt(N)."""
    N, m, n = 200, 12, 9
    A = rng.standard_normal((N, m)) * np.linspace(2.0, 0.2, m)
    W = rng.standard_normal((m, n))
    X = O.finalize_covariance(O.covariance_sum(A), N, 0.0)
    G = np.eye(n)
    Sx, Sg = O.cholesky_factors(X, G)
    Ut, s, Vt = O.whitened_svd(O.whiten(W, Sx, Sg))
    sy = np.linalg.svd(A @ W, compute_uv=False)
    np.testing.assert_allclose(s * s * N, sy * sy, rtol=1e-10)
    _, _, VyT = np.linalg.svd(A @ W)
    for k in (1, 3, 6):
        U, V = O.unwhiten(Sx, Sg, Ut, s, Vt, k)
        Vk = VyT[:k].T
        np.testing.assert_allclose(U @ V, W @ Vk @ Vk.T, atol=1e-10)


def test_identity_covariances_give_textbook_truncation():
    """X = G = I: the method is the plain truncated SVD of W (built from a known SVD)."""
    m, n = 10, 7
    P = np.linalg.qr(rng.standard_normal((m, m)))[0][:, :n]
    Q = np.linalg.qr(rng.standard_normal((n, n)))[0]
    d = np.array([9.0, 7.5, 5.0, 2.0, 1.0, 0.5, 0.25])
    W = P @ np.diag(d) @ Q.T
    Sx, Sg = O.cholesky_factors(np.eye(m), np.eye(n))
    Ut, s, Vt = O.whitened_svd(O.whiten(W, Sx, Sg))
    np.testing.assert_allclose(s, d, rtol=1e-13)
    for r in (1, 3, 7):
        U, V = O.unwhiten(Sx, Sg, Ut, s, Vt, r)
        np.testing.assert_allclose(U @ V, P[:, :r] @ np.diag(d[:r]) @ Q[:, :r].T, atol=1e-12)


def test_diagonal_covariances_closed_form():
    """Diagonal X, G and a diagonal W: W~ = sqrt(x) W sqrt(g) entry by entry, so the
    whitened singular values are |sqrt(x_i) w_i sqrt(g_i)| sorted."""
    x = np.array([4.0, 1.0, 9.0, 0.25])
    g = np.array([1.0, 16.0, 0.5, 2.0])
    w = np.array([0.5, -1.0, 0.1, 3.0])
    Sx, Sg = O.cholesky_factors(np.diag(x), np.diag(g))
    Wt = O.whiten(np.diag(w), Sx, Sg)
    np.testing.assert_allclose(Wt, np.diag(np.sqrt(x) * w * np.sqrt(g)), atol=1e-15)
    s = O.whitened_svd(Wt)[1]
    np.testing.assert_allclose(s, np.sort(np.abs(np.sqrt(x) * w * np.sqrt(g)))[::-1], rtol=1e-14)


def test_gram_route_equals_svd_route():
    for shape in ((13, 7), (7, 13), (9, 9)):
        Wt = rng.standard_normal(shape)
        s = np.linalg.svd(Wt, compute_uv=False)
        lam = O.gram_eigenvalues(Wt)
        np.testing.assert_allclose(lam, s * s, rtol=1e-10, atol=1e-12)


def test_full_rank_roundtrip():
    _, _, W, X, G = _tiny_problem(m=6, n=4, seed=11)
    Sx, Sg = O.cholesky_factors(X, G)
    Ut, s, Vt = O.whitened_svd(O.whiten(W, Sx, Sg))
    U, V = O.unwhiten(Sx, Sg, Ut, s, Vt, 4)
    np.testing.assert_allclose(U @ V, W, atol=1e-12)


# ------------------------------------------------------------------ allocation
def test_allocation_hand_cases():
    g = json.load(open(os.path.join(GOLD, "alloc_hand.json")))
    for c in g["cases"]:
        sig = [np.array(s, dtype=np.float64) for s in c["sigmas"]]
        costs = [a + b for a, b in c["mn"]]
        for prec in ("f64", "f32"):
            al = O.allocate(sig, costs, c["budget"], c["mode"], precision=prec)
            assert list(al.ranks) == c["ranks"], c
            assert al.used == c["used"]
            for got, want in ((al.cut_score, c["cut"]), (al.next_score, c["next"])):
                if want is None:
                    assert np.isnan(got)
                else:
                    assert got == want


def _walk(sigmas, costs, budget, mode):
    """Independent pure-Python statement of the sort-and-truncate walk."""
    items = []
    for u, s in enumerate(sigmas):
        for i, v in enumerate(s):
            sc = 0.5 * float(v) * float(v)
            if mode == O.KEY_PER_PARAM:
                sc /= costs[u]
            items.append((-sc, u, i))
    items.sort()
    ranks = [0] * len(sigmas)
    spent = 0
    for _, u, _ in items:
        if spent + costs[u] > budget:
            break
        spent += costs[u]
        ranks[u] += 1
    return ranks, spent


@pytest.mark.parametrize("trial", range(40))
def test_allocation_brute_force_and_invariants(trial):
    r = np.random.default_rng(trial)
    n_units = int(r.integers(1, 5))
    sig = [np.sort(r.uniform(0, 3, size=int(r.integers(1, 7))))[::-1] for _ in range(n_units)]
    if trial % 5 == 0:  # exact ties across units
        sig = [np.round(s, 1) for s in sig]
    costs = [int(r.integers(2, 12)) for _ in range(n_units)]
    total = sum(len(s) * c for s, c in zip(sig, costs))
    budget = int(r.integers(0, total + 3))
    for mode in (O.KEY_HALF_SIGMA2, O.KEY_PER_PARAM):
        al = O.allocate(sig, costs, budget, mode)
        ranks, spent = _walk(sig, costs, budget, mode)
        assert list(al.ranks) == ranks and al.used == spent
        assert spent <= budget
        kept = sum(al.ranks)
        if kept < sum(len(s) for s in sig):   # the next sorted item would overflow
            assert spent + costs[int(al.order_unit[kept])] > budget
        if mode == O.KEY_HALF_SIGMA2:
            dropped = sum(0.5 * np.sum(s[k:] ** 2) for s, k in zip(sig, al.ranks))
            assert abs(dropped - float(np.sum(al.order_score[kept:]))) <= 1e-12 * (1 + dropped)
    # information only: the greedy prefix never needs to beat the knapsack optimum
    best = 0.0
    for choice in itertools.product(*[range(len(s) + 1) for s in sig]):
        if sum(k * c for k, c in zip(choice, costs)) <= budget:
            best = max(best, sum(0.5 * np.sum(s[:k] ** 2) for s, k in zip(sig, choice)))
    al = O.allocate(sig, costs, budget, O.KEY_HALF_SIGMA2)
    greedy = sum(0.5 * np.sum(s[:k] ** 2) for s, k in zip(sig, al.ranks))
    assert greedy <= best + 1e-12


def test_allocation_sum_of_dropped_scores_is_kfac_loss():
    """Across units, the dropped scores add up to the K-FAC loss of the truncation."""
    total_dl, total_dropped = 0.0, 0.0
    res = []
    for seed in range(3):
        _, _, W, X, G = _tiny_problem(m=4 + seed, n=6 - seed, seed=seed + 20)
        Sx, Sg = O.cholesky_factors(X, G)
        Ut, s, Vt = O.whitened_svd(O.whiten(W, Sx, Sg))
        res.append((W, X, G, Sx, Sg, Ut, s, Vt))
    costs = [W.shape[0] + W.shape[1] for W, *_ in res]
    al = O.allocate([t[6] for t in res], costs, 25)
    for (W, X, G, Sx, Sg, Ut, s, Vt), k in zip(res, al.ranks):
        U, V = O.unwhiten(Sx, Sg, Ut, s, Vt, int(k))
        total_dl += O.kfac_quadratic(W - U @ V, X, G)
    total_dropped = float(np.sum(al.order_score[int(np.sum(al.ranks)):]))
    assert abs(total_dl - total_dropped) <= 1e-10 * total_dl


def test_fixed_rank_mode():
    al = O.allocate([np.ones(5), np.ones(3)], [10, 10], 0, O.FIXED_RANK, [4, 4])
    assert list(al.ranks) == [4, 3]


# ------------------------------------------------------------------------- QAW
def test_fake_quant_hand_rows():
    g = json.load(open(os.path.join(GOLD, "qaw_hand.json")))
    out = O.fake_quant_int8_token(np.array(g["rows_in"], dtype=np.float32))
    np.testing.assert_array_equal(out, np.array(g["rows_out"], dtype=np.float32))


def test_fake_quant_properties():
    A = (rng.standard_normal((64, 33)) * rng.uniform(0.01, 50, size=(64, 1))).astype(np.float32)
    Q = O.fake_quant_int8_token(A)
    s = np.abs(A).max(axis=1) / 127.0
    assert np.all(np.abs(Q - A) <= 0.5 * s[:, None] * 1.01 + np.abs(A) * 2 ** -8)
    # at most 255 levels per row, symmetric grid
    for row, sc in zip(Q, s):
        lv = np.unique(np.round(row / sc))
        assert lv.min() >= -127 and lv.max() <= 127


def test_head_units_use_the_diagonal_factor_blocks():
    """A perturbation confined to one attention head's column block (q/k/v) or row block (o)
    changes the K-FAC form only through the head's diagonal block of G (resp. X), so the
    head unit's whitened error with that block equals the full Kronecker form: LASER 2
    allocates across heads, and this is what makes a head a unit of its own."""
    r = np.random.default_rng(5)
    m, n, hd = 6, 8, 4  # two heads of width 4 on the output side
    A = r.standard_normal((60, m))
    Gr = r.standard_normal((60, n)) @ r.standard_normal((n, n))   # correlated across heads
    X = O.finalize_covariance(O.covariance_sum(A), 60, 1e-2)
    G = O.finalize_covariance(O.covariance_sum(Gr), 60, 1e-2)
    for h in range(2):
        dW = np.zeros((m, n))
        dW[:, h * hd:(h + 1) * hd] = r.standard_normal((m, hd))
        full = O.kfac_quadratic(dW, X, G)
        Sx, Sg = O.cholesky_factors(X, G[h * hd:(h + 1) * hd, h * hd:(h + 1) * hd])
        head = 0.5 * O.whitened_error(dW[:, h * hd:(h + 1) * hd], np.zeros((m, 1)), np.zeros((1, hd)), Sx, Sg)
        assert abs(full - head) <= 1e-12 * abs(full)
        # the o-side: a row block of W with the head's block of X and the full G
        dW = np.zeros((n, m))
        dW[h * hd:(h + 1) * hd, :] = r.standard_normal((hd, m))
        Xo = G  # any SPD factor on the input side
        full = O.kfac_quadratic(dW, Xo, X)
        Sx, Sg = O.cholesky_factors(Xo[h * hd:(h + 1) * hd, h * hd:(h + 1) * hd], X)
        head = 0.5 * O.whitened_error(dW[h * hd:(h + 1) * hd, :], np.zeros((hd, 1)), np.zeros((1, m)), Sx, Sg)
        assert abs(full - head) <= 1e-12 * abs(full)
    # the oracle's whole-workload run takes exactly those blocks for head units
    from synth import recipes
    wl = recipes.mini_vlm(n_tokens=64)
    ids = [i for i, u in enumerate(wl.units) if u.name in ("lm.b0.q.h1", "lm.b0.o.h1")]
    res = O.compress_workload(wl, units=ids)
    for ur, i in zip(res["units"], ids):
        u = wl.units[i]
        Xf = res["covs"][u.x_site]
        Gf = res["covs"][u.g_site]
        np.testing.assert_array_equal(ur.X, Xf[u.x_off:u.x_off + u.m, u.x_off:u.x_off + u.m])
        np.testing.assert_array_equal(ur.G, Gf[u.g_off:u.g_off + u.n, u.g_off:u.g_off + u.n])
        np.testing.assert_array_equal(ur.Wt, O.whiten(recipes.gen_full_weight(wl, u)[
            u.row0:u.row0 + u.m, u.col0:u.col0 + u.n], ur.Sx, ur.Sg))


def test_energy_ratio_key_unirank():
    """UniRank 2.1: s_{l,i} = I_l sigma_{l,i}^2 / ||Sigma_l||_F^2, sorted and truncated under the
    m + n cost of each kept pair."""
    # hand case: unit 0 sigma (2, 1) -> energy 5 -> keys 0.8, 0.2; unit 1 sigma (1, 1) ->
    # keys 0.5, 0.5; costs 10 each.  Sorted: 0.8 (u0), 0.5 (u1), 0.5 (u1), 0.2 (u0).
    sig = [np.array([2.0, 1.0]), np.array([1.0, 1.0])]
    al = O.allocate(sig, [10, 10], 30, O.KEY_ENERGY_RATIO)
    assert list(al.ranks) == [1, 2] and al.used == 30 and abs(al.cut_score - 0.5) < 1e-15
    # weights I = (1, 2): unit 1's keys become 1.0, 1.0, ahead of 0.8; budget 20 keeps only them
    al = O.allocate(sig, [10, 10], 20, O.KEY_ENERGY_RATIO, weights=[1.0, 2.0])
    assert list(al.ranks) == [0, 2] and abs(al.cut_score - 1.0) < 1e-15 and abs(al.next_score - 0.8) < 1e-15
    # a zero weight removes a unit from the competition
    al = O.allocate(sig, [10, 10], 40, O.KEY_ENERGY_RATIO, weights=[0.0, 1.0])
    assert list(al.ranks) == [2, 2] and al.order_unit[-1] == 0
    r = np.random.default_rng(11)
    sigs = [np.sort(r.gamma(1.0, 1.0, k))[::-1] for k in (9, 14, 6)]
    costs = [30, 25, 17]
    budget = 300
    # one unit alone: a positive multiple of sigma^2, so the same ranks as 1/2 sigma^2
    for s_ in sigs:
        assert list(O.allocate([s_], [20], 100, O.KEY_ENERGY_RATIO).ranks) == \
            list(O.allocate([s_], [20], 100, O.KEY_HALF_SIGMA2).ranks)
    # invariant to rescaling a unit's spectrum (1/2 sigma^2 is not)
    base = O.allocate(sigs, costs, budget, O.KEY_ENERGY_RATIO).ranks
    scaled = [sigs[0] * 10.0] + sigs[1:]
    assert list(O.allocate(scaled, costs, budget, O.KEY_ENERGY_RATIO).ranks) == list(base)
    assert list(O.allocate(scaled, costs, budget, O.KEY_HALF_SIGMA2).ranks) != \
        list(O.allocate(sigs, costs, budget, O.KEY_HALF_SIGMA2).ranks)
    # weights multiply: w = 1 everywhere changes nothing, a common factor changes nothing
    assert list(O.allocate(sigs, costs, budget, O.KEY_ENERGY_RATIO, weights=[1, 1, 1]).ranks) == list(base)
    assert list(O.allocate(sigs, costs, budget, O.KEY_ENERGY_RATIO, weights=[3, 3, 3]).ranks) == list(base)
    # the float32 evaluation ranks like the float64 one away from ties
    assert list(O.allocate(sigs, costs, budget, O.KEY_ENERGY_RATIO, precision="f32",
                           weights=[0.5, 2.0, 1.0]).ranks) == \
        list(O.allocate(sigs, costs, budget, O.KEY_ENERGY_RATIO, weights=[0.5, 2.0, 1.0]).ranks)


def test_empirical_fisher_score_is_the_rank_one_fisher_form():
    """LASER 2: the empirical-Fisher score of component i is 1/2 vec(dW)^T F vec(dW) for
    dW = u_i v_i, with F the explicit empirical Fisher (1/N) sum_t g_t g_t^T over the
    per-token weight gradients g_t = vec(a_t^T gr_t) (column-major vec, d_in x d_out)."""
    r = np.random.default_rng(21)
    N, m, n, k = 40, 4, 5, 3
    A = r.standard_normal((N, m))
    Gr = r.standard_normal((N, n))
    U = r.standard_normal((m, k))
    V = r.standard_normal((k, n))
    F = np.zeros((m * n, m * n))
    for t in range(N):
        g = np.outer(A[t], Gr[t]).reshape(-1, order="F")
        F += np.outer(g, g) / N
    sc = O.empirical_fisher_scores(A, Gr, U, V)
    for i in range(k):
        dw = np.outer(U[:, i], V[i]).reshape(-1, order="F")
        assert abs(sc[i] - 0.5 * dw @ F @ dw) <= 1e-12 * abs(sc[i])
    # when the gradients are a fixed direction times a scalar independent of the activation
    # amplitudes... the K-FAC factorisation is exact, F = G kron X, and the score is
    # 1/2 (u^T X u)(v G v^T); with the whitened factors this is 1/2 sigma^2
    c = r.standard_normal(N)
    d = r.standard_normal(n)
    Gr1 = np.outer(np.ones(N), d)             # g_t = d for every token: G = d d^T
    X = A.T @ A / N
    Gm = np.outer(d, d)
    sc = O.empirical_fisher_scores(A, Gr1, U, V)
    for i in range(k):
        assert abs(sc[i] - 0.5 * (U[:, i] @ X @ U[:, i]) * (V[i] @ Gm @ V[i])) <= 1e-10 * abs(sc[i])


def test_allocate_keys_matches_monotone_allocation_and_selects_subsets():
    r = np.random.default_rng(22)
    sigs = [np.sort(r.gamma(1.0, 1.0, k))[::-1] for k in (8, 11, 5)]
    costs = [13, 21, 9]
    for budget in (0, 50, 150, 10 ** 6):
        a = O.allocate(sigs, costs, budget)
        b = O.allocate_keys([0.5 * s * s for s in sigs], costs, budget)
        assert list(a.ranks) == list(b.ranks) and a.used == b.used
    keys = [np.array([0.1, 0.9, 0.5]), np.array([0.7, 0.2])]
    al = O.allocate_keys(keys, [10, 10], 30)      # keeps 0.9 (u0 c1), 0.7 (u1 c0), 0.5 (u0 c2)
    assert list(al.ranks) == [2, 1]
    assert sorted(zip(al.order_unit[:3], al.order_comp[:3])) == [(0, 1), (0, 2), (1, 0)]


def test_swift_closed_form_hand_case():
    """Swift-SVD 2A on a hand case: A = [[2, 0], [0, 1]], W = I: C = diag(2, 0.5), sigma =
    (sqrt 2, sqrt 0.5), W_1 = diag(1, 0), loss (1/N)||A (W - W_1)||^2 = 0.5 = lambda_2."""
    A = np.array([[2.0, 0.0], [0.0, 1.0]])
    W = np.eye(2)
    C = O.output_covariance(A, W)
    np.testing.assert_array_equal(C, np.diag([2.0, 0.5]))
    sig, V = O.output_eig(C)
    np.testing.assert_allclose(sig, [np.sqrt(2.0), np.sqrt(0.5)], rtol=1e-15)
    U, Vt = O.activation_factors(W, V, 1)
    np.testing.assert_allclose(np.abs(U @ Vt), np.diag([1.0, 0.0]), atol=1e-15)
    assert abs(O.activation_loss(A, W, U, Vt) - 0.5) < 1e-15


@pytest.mark.parametrize("shape", [(60, 6, 5), (60, 4, 7), (3, 5, 6)])
def test_swift_closed_form_is_the_activation_aware_optimum(shape):
    """Swift-SVD 2A: W V_k V_k^T minimises ||A W - A W_k||; its loss is the sum of the dropped
    eigenvalues of C, equals the Eckart-Young optimum of Y = A W (library SVD of Y, not the
    eigendecomposition), and no random rank-k candidate does better.  The last shape has
    N < m (rank-deficient activations, where a Cholesky of X would fail)."""
    N, m, n = shape
    r = np.random.default_rng(N * 100 + m * 10 + n)
    A = r.standard_normal((N, m)) * np.linspace(3.0, 0.2, m)[None, :]
    W = r.standard_normal((m, n))
    sig, V = O.output_eig(O.output_covariance(A, W))
    y_sv = np.linalg.svd(A @ W, compute_uv=False)
    for k in range(0, min(m, n) + 1):
        U, Vt = O.activation_factors(W, V, k)
        loss = O.activation_loss(A, W, U, Vt)
        assert abs(loss - np.sum(sig[k:] ** 2)) <= 1e-10 * max(1.0, np.sum(sig ** 2))
        assert abs(loss - np.sum(y_sv[k:] ** 2) / N) <= 1e-10 * max(1.0, np.sum(sig ** 2))
        for _ in range(50):
            Ur = r.standard_normal((m, k))
            Vr = r.standard_normal((k, n))
            assert O.activation_loss(A, W, Ur, Vr) >= loss - 1e-9
            P = np.linalg.qr(r.standard_normal((n, n)))[0][:, :k]
            assert O.activation_loss(A, W, W @ P, P.T) >= loss - 1e-9


def test_swift_route_is_the_whitened_path_with_identity_gradient_factor():
    """With G = I and no damping the whitened path computes the same thing: S_x^T S_x = X
    gives W~^T W~ = W^T X W = C, so the whitened singular values equal Swift's sigma and
    the unwhitened rank-k product S_x^-1 U~_k Sigma_k V~_k^T equals W V_k V_k^T."""
    r = np.random.default_rng(31)
    N, m, n = 80, 7, 5
    A = r.standard_normal((N, m))
    W = r.standard_normal((m, n))
    X = O.finalize_covariance(O.covariance_sum(A), N, 0.0)
    np.testing.assert_allclose(W.T @ X @ W, O.output_covariance(A, W), rtol=1e-12, atol=1e-12)
    Sx, Sg = O.cholesky_factors(X, np.eye(n))
    Ut, s, Vt = O.whitened_svd(O.whiten(W, Sx, Sg))
    sig, V = O.output_eig(O.output_covariance(A, W))
    np.testing.assert_allclose(s, sig[:len(s)], rtol=1e-10)
    for k in range(0, n + 1):
        U1, V1 = O.unwhiten(Sx, Sg, Ut, s, Vt, k)
        U2, V2 = O.activation_factors(W, V, k)
        np.testing.assert_allclose(U1 @ V1, U2 @ V2, atol=1e-10)


def test_swift_output_covariance_aggregates_by_chunks():
    """Swift-SVD 2A's incremental aggregation: token chunks summed give the whole covariance."""
    r = np.random.default_rng(32)
    A = r.standard_normal((37, 6))
    W = r.standard_normal((6, 4))
    parts = sum(O.output_covariance(A[t:t + 10], W) * len(A[t:t + 10]) for t in range(0, 37, 10)) / 37
    np.testing.assert_allclose(parts, O.output_covariance(A, W), rtol=1e-13, atol=1e-13)


def test_channel_errors_are_the_per_channel_mean_squared_preactivation_error():
    """LASER hybrid FFN: with X = A^T A / N the error of channel j is (1/N) sum_t
    (a_t . (w_j - w^_j))^2, checked token by token; summed over the channels and with
    X = S_x^T S_x it is ||S_x (W - U V)||_F^2, the whitened error with G = I."""
    r = np.random.default_rng(51)
    N, d, f, k = 30, 5, 7, 2
    A = r.standard_normal((N, d))
    W = r.standard_normal((d, f))
    U = r.standard_normal((d, k))
    V = r.standard_normal((k, f))
    X = A.T @ A / N
    e = O.channel_errors(W, U, V, X)
    D = W - U @ V
    for j in range(f):
        want = np.mean([(A[t] @ D[:, j]) ** 2 for t in range(N)])
        assert abs(e[j] - want) <= 1e-12 * max(1.0, want)
    Sx, _ = O.cholesky_factors(X, np.eye(f))
    assert abs(e.sum() - O.whitened_error(W, U, V, Sx, np.eye(f))) <= 1e-10 * e.sum()


def test_svd_friendly_channels_hand_case():
    """Channels inside the span of the temporary factors reconstruct exactly and are chosen;
    equal errors leave the lower channel indices dense."""
    d = 4
    u = np.array([[1.0], [0.0], [0.0], [0.0]])
    W = np.zeros((d, 5))
    W[:, 1] = 3.0 * u[:, 0]          # in span(u): error 0
    W[:, 3] = -2.0 * u[:, 0]         # in span(u): error 0
    W[:, 0] = [0.0, 1.0, 0.0, 0.0]   # orthogonal: error 1 (X = I)
    W[:, 2] = [0.0, 0.0, 2.0, 0.0]   # error 4
    W[:, 4] = [0.5, 0.0, 0.0, 0.5]   # error 0.25
    V = u.T @ W                      # U V = u u^T W: the projection of W onto span(u)
    e = O.channel_errors(W, u, V, np.eye(d))
    np.testing.assert_allclose(e, [1.0, 0.0, 4.0, 0.0, 0.25], atol=1e-15)
    np.testing.assert_array_equal(O.select_svd_channels([e], 2), [1, 3])
    np.testing.assert_array_equal(O.select_svd_channels([e], 3), [1, 3, 4])
    # gate and up share the channel: the errors add
    e_up = np.array([0.0, 5.0, 0.0, 0.0, 0.0])
    np.testing.assert_array_equal(O.select_svd_channels([e, e_up], 2), [3, 4])
    # ties: the lower indices stay dense
    np.testing.assert_array_equal(O.select_svd_channels([np.zeros(5)], 3), [2, 3, 4])
    np.testing.assert_array_equal(O.select_svd_channels([e], 0), [])
    np.testing.assert_array_equal(O.select_svd_channels([e], 5), [0, 1, 2, 3, 4])


def test_hybrid_ffn_flow_accounting_and_limits():
    """LASER hybrid FFN over a small block: the split covers every hidden channel once; the
    dense channels' cost comes off the budget; with every channel SVD-friendly the SVD branch
    is the ordinary gate/up whitened SVD (same spectra as the plain path); with none, gate and
    up are dense and only the other units compete for what is left."""
    from synth import recipes
    wl = recipes.mini_block(n_tokens=300, d=64, ffn=96, kv=32, seed=5)
    f = 96
    out = O.compress_hybrid_ffn(wl, r_temp=8, n_svd=40)
    sp = out["splits"][0]
    assert sorted(np.concatenate([sp["svd"], sp["dense"]]).tolist()) == list(range(f))
    assert len(sp["svd"]) == 40
    assert out["dense_cost"] == 2 * 64 * (f - 40)
    assert out["budget"] == wl.budget - out["dense_cost"]
    used = sum(e[2].rank * (e[2].m + e[2].n) for e in out["entries"])
    assert used == out["alloc"].used <= out["budget"]
    # all channels SVD-friendly: the branch is the plain path's gate and up
    full = O.compress_hybrid_ffn(wl, r_temp=8, n_svd=f)
    plain = O.compress_workload(wl)
    names = [u.name for u in wl.units]
    for kind, i, r in full["entries"]:
        if kind == "svd":
            np.testing.assert_allclose(r.sigma, plain["units"][i].sigma, rtol=1e-10, atol=1e-12)
    # no channel SVD-friendly: gate and up contribute no entry
    none = O.compress_hybrid_ffn(wl, r_temp=8, n_svd=0)
    assert all(kind == "unit" for kind, _, _ in none["entries"])
    assert {names[i] for _, i, _ in none["entries"]} == set(names) - {"gate", "up"}


def test_swift_hybrid_keys_hand_case():
    """Swift-SVD B hybrid scoring as per-component keys, on a hand-worked case
    (tests/golden/swift_hybrid_hand.json): the keys, and the sort-and-truncate over them."""
    g = json.load(open(os.path.join(GOLD, "swift_hybrid_hand.json")))
    for s, b, want in zip(g["sigmas"], g["betas"], g["keys"]):
        got = O.swift_hybrid_keys(np.array(s, dtype=np.float32), b, g["alpha"])
        assert got.dtype == np.float32
        np.testing.assert_allclose(got.astype(np.float64), want, rtol=1e-7, atol=0)
    for c in g["cases"]:
        al = O.allocate_swift_hybrid([np.array(s, np.float32) for s in g["sigmas"]], g["costs"], c["budget"],
                                     g["betas"], g["alpha"])
        assert list(al.ranks) == c["ranks"] and al.used == c["used"]
        for got, want in ((al.cut_score, c["cut"]), (al.next_score, c["next"])):
            if want is None:
                assert np.isnan(got)
            else:
                assert abs(got - want) <= 1e-7 * abs(want)


def test_swift_residual_loss_is_the_truncation_loss():
    """eps*_k (Swift-SVD B's closed-form loss at rank k) equals the whitened error of the
    rank-k factors mapped back, ||S_x (W - U_k V_k) S_g||^2 (Swift-SVD 2A / LASER 1 optimum),
    for every k, and is non-increasing with eps*_0 = ||W~||_F^2."""
    A, Gr, W, X, G = _tiny_problem(m=6, n=5, N=40, seed=3)
    Sx, Sg = O.cholesky_factors(X, G)
    Ut, s, Vt = O.whitened_svd(O.whiten(W, Sx, Sg))
    s32 = s.astype(np.float32)
    eps = O.swift_residual_losses(s32)
    assert all(eps[k] >= eps[k + 1] for k in range(len(eps) - 1))
    for k in range(len(s)):
        U, V = O.unwhiten(Sx, Sg, Ut, s, Vt, k)
        e = O.whitened_error(W, U, V, Sx, Sg)
        assert abs(eps[k] - e) <= 1e-6 * eps[0] + 1e-12, k
    assert abs(eps[0] - float(np.sum(O.whiten(W, Sx, Sg) ** 2))) <= 1e-6 * eps[0]


def test_swift_hybrid_limits_and_monotone_keys():
    """alpha = 1: the key is beta alone, so units are filled whole in decreasing beta (ties to
    the lower unit).  alpha = 0: the key is log(e + eps*), a monotone map of the residual
    loss, so the allocation equals sorting by eps* itself.  Any alpha: keys non-increasing
    along a unit (the kept set is a prefix); beta <= 0 gives keys 0."""
    r = np.random.default_rng(31)
    sigs = [np.sort(r.gamma(1.0, 1.0, k)).astype(np.float32)[::-1].copy() for k in (6, 9, 4)]
    costs = [11, 15, 7]
    betas = [0.5, 2.0, 1.0]
    total = sum(c * len(s) for c, s in zip(costs, sigs))
    for budget in (0, 40, 100, 160, total):
        al = O.allocate_swift_hybrid(sigs, costs, budget, betas, 1.0)
        want, left = [0, 0, 0], budget
        for u in (1, 2, 0):
            k = min(len(sigs[u]), left // costs[u])
            want[u] = k
            if k < len(sigs[u]):
                break
            left -= k * costs[u]
        assert list(al.ranks) == want, (budget, list(al.ranks), want)
        a0 = O.allocate_swift_hybrid(sigs, costs, budget, betas, 0.0)
        e0 = O.allocate_keys([np.array(O.swift_residual_losses(s)) for s in sigs], costs, budget)
        assert list(a0.ranks) == list(e0.ranks)
    for alpha in (0.0, 0.3, 0.7, 1.0):
        for s, b in zip(sigs, betas):
            k = O.swift_hybrid_keys(s, b, alpha)
            assert np.all(np.diff(k.astype(np.float64)) <= 0)
    assert not np.any(O.swift_hybrid_keys(sigs[0], 0.0, 0.5))
    assert not np.any(O.swift_hybrid_keys(sigs[0], -1.0, 0.5))


def test_swift_hybrid_allocation_is_the_greedy_next_component_rule():
    """The sort-and-truncate over the hybrid keys is the greedy process the reading states:
    repeatedly give the next component to the unit whose current truncation has the highest
    hybrid score (recomputed from the dropped components' energy), ties to the lower unit, and
    stop at the first component that would overflow the budget."""
    r = np.random.default_rng(44)
    for trial in range(20):
        nu = int(r.integers(1, 5))
        sigs = [np.sort(r.gamma(0.7, 1.0, int(r.integers(1, 7)))).astype(np.float32)[::-1].copy()
                for _ in range(nu)]
        costs = [int(r.integers(1, 9)) for _ in range(nu)]
        betas = [float(r.uniform(0.1, 3.0)) for _ in range(nu)]
        alpha = float(r.uniform(0.0, 1.0))
        budget = int(r.integers(0, 60))
        held, spent = [0] * nu, 0
        while True:
            best, bu = None, -1
            for u in range(nu):
                if held[u] == len(sigs[u]):
                    continue
                rest = sum(float(x) * float(x) for x in sigs[u][held[u]:].astype(np.float64))
                sc = float(np.float32(betas[u] ** alpha * np.log(np.e + rest) ** (1.0 - alpha)))
                if best is None or sc > best:
                    best, bu = sc, u
            if bu < 0 or spent + costs[bu] > budget:
                break
            held[bu] += 1
            spent += costs[bu]
        al = O.allocate_swift_hybrid(sigs, costs, budget, betas, alpha)
        assert list(al.ranks) == held and al.used == spent, trial


def test_hybrid_ffn_budget():
    """LASER hybrid FFN: the dense channels' parameters come off the budget first (d_model
    weights per dense channel and projection); never below zero."""
    assert O.hybrid_ffn_budget(1000, [64, 64], [3, 3]) == 1000 - 384
    assert O.hybrid_ffn_budget(100, [64, 64], [3, 3]) == 0
    assert O.hybrid_ffn_budget(500, [], []) == 500
