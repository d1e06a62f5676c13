"""GPU parity: every step of the path, called through the C ABI, against the fp64 oracle
on the same seeded inputs (small shapes spanning several tiles and ragged tails).

Tolerances (stated by the hot-path contract): covariances relative Frobenius <= 1e-4;
singular values |sigma - sigma_oracle| <= 1e-3 sigma_max per unit; whitened-error ratio
|e / e_opt - 1| <= 1e-3; ranks identical for identical float32 sigma, and end to end
identical except at score ties (within 1e-6 of the cut); integer work bit-exact.
"""
import numpy as np
import pytest

import oracle as O
from synth import recipes
from tests.gpu_util import bf16_dev, lower, rank_parity, rel_fro, to_dev

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def ctx():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from vlm_compression_fac_b300 import kfsvd as K
    c = K.Context(0)
    yield c
    c.close()


def K():
    from vlm_compression_fac_b300 import kfsvd
    return kfsvd


# ------------------------------------------------------------------ generator
def test_device_generator_matches_host():
    from synth import device
    for wl, site in ((recipes.mini_block(), "down_in"), (recipes.single_linear(), "in"),
                     (recipes.mini_block(), "q_out")):
        s = wl.sites[site]
        dev = device.stream_on_device(wl, s, 0, 300, torch).float().cpu().numpy()
        host = recipes.gen_stream(wl, s, 0, 300)
        np.testing.assert_array_equal(dev, host)
    wl = recipes.mini_block()
    u = wl.units[4]
    np.testing.assert_array_equal(device.weight_on_device(wl, u, torch).float().cpu().numpy(),
                                  recipes.gen_weight(wl, u))


# ------------------------------------------------------------------ step 1
@pytest.mark.parametrize("d,n_tok", [(320, 1000), (704, 777), (128, 64), (256, 4097)])
def test_kfac_accumulate_bf16(ctx, d, n_tok):
    wl = recipes.mini_block(n_tokens=n_tok, d=d, ffn=704)
    A = recipes.gen_stream(wl, wl.sites["attn_in"], 0, n_tok)
    cov = torch.full((d, d), 7.0, dtype=torch.float32, device="cuda")
    cov.copy_(torch.tril(torch.zeros_like(cov)) + torch.triu(torch.full_like(cov, 7.0), 1))
    half = n_tok // 2
    Ad = bf16_dev(A, torch)
    K().kfac_accumulate(ctx, Ad[:half], cov)
    K().kfac_accumulate(ctx, Ad[half:], cov)
    ctx.sync_status()
    got = cov.cpu().numpy()
    want = O.covariance_sum(A)
    assert rel_fro(lower(got), lower(want)) <= 1e-4
    assert np.all(np.triu(got, 1) == np.triu(np.full((d, d), 7.0, np.float32), 1))


@pytest.mark.parametrize("site", ["in", "out"])
def test_kfac_accumulate_f32_single_linear(ctx, site):
    wl = recipes.single_linear()
    A = recipes.gen_stream(wl, wl.sites[site], 0, wl.n_tokens)
    d = A.shape[1]
    cov = torch.zeros((d, d), dtype=torch.float32, device="cuda")
    K().kfac_accumulate(ctx, to_dev(A, torch), cov)
    ctx.sync_status()
    assert rel_fro(lower(cov.cpu().numpy()), lower(O.covariance_sum(A))) <= 1e-4


def test_fake_quant_is_bit_exact(ctx):
    """One token per call: the diagonal of the sum is exactly the squared quantised value."""
    wl = recipes.mini_block(n_tokens=48, d=320)
    A = recipes.gen_stream(wl, wl.sites["attn_in"], 0, 48)
    A[5] = 0.0                         # zero row stays zero
    A[7, 3] = -np.abs(A[7]).max() * 2  # amax in a negative entry
    A = recipes.philox.bf16_bits_to_f32(recipes.philox.f32_to_bf16_bits(A))
    Q = O.fake_quant_int8_token(A)
    Ad = bf16_dev(A, torch)
    for t in range(A.shape[0]):
        cov = torch.zeros((320, 320), dtype=torch.float32, device="cuda")
        K().kfac_accumulate(ctx, Ad[t:t + 1], cov, quant=K().KF_QUANT_INT8_TOKEN)
        diag = torch.diagonal(cov).cpu().numpy()
        np.testing.assert_array_equal(diag, (Q[t].astype(np.float32) ** 2).astype(np.float32))
        first = cov[:, 0].cpu().numpy()    # column 0 of the lower triangle: q_i * q_0
        np.testing.assert_array_equal(first, (Q[t] * Q[t][0]).astype(np.float32))
    ctx.sync_status()


def test_kfac_accumulate_qaw_covariance(ctx):
    wl = recipes.mini_block(n_tokens=1000, quant="int8_token")
    A = recipes.gen_stream(wl, wl.sites["mlp_in"], 0, 1000)
    cov = torch.zeros((320, 320), dtype=torch.float32, device="cuda")
    K().kfac_accumulate(ctx, bf16_dev(A, torch), cov, quant=K().KF_QUANT_INT8_TOKEN)
    ctx.sync_status()
    want = O.covariance_sum(O.fake_quant_int8_token(A))
    assert rel_fro(lower(cov.cpu().numpy()), lower(want)) <= 1e-4


def test_finalize(ctx):
    wl = recipes.mini_block(n_tokens=500)
    A = recipes.gen_stream(wl, wl.sites["down_in"], 0, 500)
    S = np.tril(O.covariance_sum(A)).astype(np.float32)
    cov = to_dev(S, torch)
    K().kf_finalize_covariance(ctx, cov, 500, 1e-2)
    ctx.sync_status()
    want = O.finalize_covariance(np.tril(S) + np.tril(S, -1).T, 500, 1e-2)
    got = cov.cpu().numpy()
    assert rel_fro(got, want) <= 1e-6
    np.testing.assert_array_equal(got, got.T)


# ------------------------------------------------------------ steps 2 and 3
def _factors(m, n, seed, n_tok=1500):
    wl = recipes.mini_block(n_tokens=n_tok, d=m, ffn=max(m, n), kv=n, seed=seed)
    A = recipes.gen_stream(wl, recipes.Site("a", m, "act"), 0, n_tok)
    Gr = recipes.gen_stream(wl, recipes.Site("g", n, "grad"), 0, n_tok)
    X = O.finalize_covariance(O.covariance_sum(A), n_tok, 1e-2).astype(np.float32)
    G = O.finalize_covariance(O.covariance_sum(Gr), n_tok, 1e-2).astype(np.float32)
    W = recipes.gen_weight(wl, recipes.Unit("w", m, n, "a", "g"))
    return X, G, W


def _gpu_whiten(ctx, X, G, W):
    m, n = W.shape
    s = min(m, n)
    Sx = torch.empty((m, m), dtype=torch.float32, device="cuda")
    Sg = torch.empty((n, n), dtype=torch.float32, device="cuda")
    Si = torch.empty((s, s), dtype=torch.float32, device="cuda")
    Wt = torch.empty((m, n), dtype=torch.float32, device="cuda")
    K().whiten(ctx, to_dev(X, torch), to_dev(G, torch), bf16_dev(W, torch), Sx, Sg, Si, Wt)
    ctx.sync_status()
    return Sx, Sg, Si, Wt


@pytest.mark.parametrize("m,n", [(320, 192), (320, 704), (704, 320), (257, 257), (64, 130)])
def test_whiten(ctx, m, n):
    X, G, W = _factors(m, n, seed=m * 7 + n)
    Sx, Sg, Si, Wt = _gpu_whiten(ctx, X, G, W)
    oSx, oSg = O.cholesky_factors(X.astype(np.float64), G.astype(np.float64))
    assert rel_fro(Sx.cpu().numpy(), oSx) <= 1e-5
    assert rel_fro(Sg.cpu().numpy(), oSg) <= 1e-5
    assert np.all(np.tril(Sx.cpu().numpy(), -1) == 0) and np.all(np.triu(Sg.cpu().numpy(), 1) == 0)
    inv = np.linalg.inv(oSg) if n <= m else np.linalg.inv(oSx)
    assert rel_fro(Si.cpu().numpy(), inv) <= 1e-4
    assert rel_fro(Wt.cpu().numpy(), O.whiten(W, oSx, oSg)) <= 1e-5


@pytest.mark.parametrize("sizes", [(320, 704, 192), (1000, 64, 257), (513,)])
def test_factor_covariances_batched(ctx, sizes):
    """Step 2 for several factors at once (independent chains on the context's streams):
    each S = chol_lower(A) or its transpose (relative Frobenius 1e-5), and its inverse
    (1e-4, as in the whitening test: the float32 rounding of A alone moves S^-1 by about
    u kappa(S), 3e-6 .. 7e-6 for these factors with kappa 50 .. 120), against float64 LAPACK on
    the same damped factors; sizes below, at and across the 256-wide column strips and the
    doubling levels of the inverse."""
    r = np.random.default_rng(sum(sizes))
    jobs, want = [], []
    for j, n in enumerate(sizes):
        B = r.standard_normal((n + 40, n)) * (1.0 / np.sqrt(np.arange(1, n + 1)))
        A = O.finalize_covariance(O.covariance_sum(B), n + 40, 1e-2).astype(np.float32)
        upper = j % 2 == 1
        S = torch.empty((n, n), dtype=torch.float32, device="cuda")
        Si = torch.empty((n, n), dtype=torch.float32, device="cuda")
        jobs.append((to_dev(A, torch), S, Si, upper))
        L = np.linalg.cholesky(A.astype(np.float64))
        F = L.T if upper else L
        want.append((F, np.linalg.inv(F)))
    K().factor_covariances(ctx, jobs)
    ctx.sync_status()
    for (A, S, Si, upper), (F, Fi) in zip(jobs, want):
        assert rel_fro(S.cpu().numpy(), F) <= 1e-5
        assert rel_fro(Si.cpu().numpy(), Fi) <= 1e-4


def test_whiten_not_spd_reports_pivot(ctx):
    X = np.eye(96, dtype=np.float32)
    X[40, 40] = -1.0
    G = np.eye(64, dtype=np.float32)
    W = np.zeros((96, 64), dtype=np.float32)
    Sx = torch.empty((96, 96), device="cuda")
    Sg = torch.empty((64, 64), device="cuda")
    Si = torch.empty((64, 64), device="cuda")
    Wt = torch.empty((96, 64), device="cuda")
    K().whiten(ctx, to_dev(X, torch), to_dev(G, torch), to_dev(W, torch), Sx, Sg, Si, Wt)
    with pytest.raises(K().KfsvdError) as e:
        ctx.sync_status()
    assert e.value.status == K().KF_ERR_NOT_SPD and "info 40" in str(e.value)
    ctx.sync_status()  # cleared


# ------------------------------------------------------------------ step 4
def _gpu_svd(ctx, Wts, tol=1e-6, max_sweeps=30):
    s = min(Wts[0].shape)
    sig = [torch.empty(s, device="cuda") for _ in Wts]
    vec = [torch.empty((s, s), device="cuda") for _ in Wts]
    sw = torch.zeros(len(Wts), dtype=torch.int32, device="cuda")
    K().whitened_svd(ctx, [to_dev(w.astype(np.float32), torch) for w in Wts], sig, vec, sweeps=sw, tol=tol,
                     max_sweeps=max_sweeps)
    ctx.sync_status()
    return [x.cpu().numpy() for x in sig], [v.cpu().numpy() for v in vec], sw.cpu().numpy()


@pytest.mark.parametrize("shapes", [[(320, 192)], [(192, 320)], [(257, 300)], [(64, 64)],
                                    [(320, 192), (192, 600), (700, 192)]])
def test_whitened_svd(ctx, shapes):
    Wts = []
    for i, (m, n) in enumerate(shapes):
        X, G, W = _factors(m, n, seed=11 + i)
        oSx, oSg = O.cholesky_factors(X.astype(np.float64), G.astype(np.float64))
        Wts.append(O.whiten(W, oSx, oSg))
    sig, vec, sweeps = _gpu_svd(ctx, Wts)
    for Wt, s_g, V, sw in zip(Wts, sig, vec, sweeps):
        s_o = O.whitened_svd(Wt.astype(np.float32).astype(np.float64))[1]
        assert np.all(np.diff(s_g) <= 0)
        assert np.max(np.abs(s_g - s_o)) <= 1e-3 * s_o[0]
        assert 1 <= sw <= 30
        # unit-norm, mutually orthogonal columns
        assert np.max(np.abs(V.T.astype(np.float64) @ V - np.eye(V.shape[0]))) <= 2e-4
        m, n = Wt.shape
        C = Wt.T @ Wt if n <= m else Wt @ Wt.T
        R = C @ V - V * (s_g.astype(np.float64) ** 2)[None, :]
        assert np.linalg.norm(R) <= 1e-3 * np.linalg.norm(C)


def test_whitened_svd_reports_no_convergence(ctx):
    X, G, W = _factors(256, 256, seed=5)
    oSx, oSg = O.cholesky_factors(X.astype(np.float64), G.astype(np.float64))
    s = torch.empty(256, device="cuda")
    v = torch.empty((256, 256), device="cuda")
    K().whitened_svd(ctx, [to_dev(O.whiten(W, oSx, oSg).astype(np.float32), torch)], [s], [v], max_sweeps=1)
    with pytest.raises(K().KfsvdError) as e:
        ctx.sync_status()
    assert e.value.status == K().KF_ERR_NO_CONVERGENCE


# ---------------------------------------------------------------- step 5a
def _gpu_alloc(ctx, sigmas, costs, budget, mode, fixed=None):
    sig = torch.from_numpy(np.concatenate(sigmas).astype(np.float32)).cuda()
    off = torch.tensor([0] + list(np.cumsum([len(s) for s in sigmas])), dtype=torch.int64, device="cuda")
    cost = torch.tensor(costs, dtype=torch.int64, device="cuda")
    ranks = torch.empty(len(sigmas), dtype=torch.int32, device="cuda")
    cut = torch.empty(2, dtype=torch.float32, device="cuda")
    used = torch.zeros(1, dtype=torch.int64, device="cuda")
    fr = None if fixed is None else torch.tensor(fixed, dtype=torch.int32, device="cuda")
    K().score_and_allocate(ctx, sig, off, cost, budget, ranks, mode=mode, fixed_rank=fr, cut=cut, used=used)
    ctx.sync_status()
    return ranks.cpu().numpy(), cut.cpu().numpy(), int(used.item())


ALLOC_CASES = [
    # (n_units, max_len, budget_fraction, mode, ties)
    (7, 400, 0.5, "half_sigma2", False),
    (7, 400, 0.3, "per_param", False),
    (12, 64, 0.4, "half_sigma2", True),
    (100, 4000, 0.4, "half_sigma2", False),   # ~200k keys: many radix tiles
    (3, 10, 0.0, "half_sigma2", False),
    (3, 10, 2.0, "half_sigma2", False),
    (300, 4100, 0.37, "per_param", True),     # ~600k keys
]


@pytest.mark.parametrize("case", ALLOC_CASES)
def test_allocation_bit_identical(ctx, case):
    nu, ml, frac, mode, ties = case
    r = np.random.default_rng(nu * 1000 + ml)
    sig, costs = [], []
    for u in range(nu):
        m, n = int(r.integers(8, ml + 8)), int(r.integers(8, ml + 8))
        s = np.sort(r.gamma(1.0, 1.0, size=min(m, n)))[::-1].astype(np.float32)
        if ties:
            s = np.round(s, 2).astype(np.float32)
        sig.append(s)
        costs.append(m + n)
    budget = int(frac * sum(len(s) * c for s, c in zip(sig, costs)))
    kmode = K().KF_KEY_PER_PARAM if mode == "per_param" else K().KF_KEY_HALF_SIGMA2
    ranks, cut, used = _gpu_alloc(ctx, sig, costs, budget, kmode)
    al = O.allocate(sig, costs, budget, mode, precision="f32")
    np.testing.assert_array_equal(ranks, al.ranks)
    assert used == al.used
    for g, w in zip(cut, (al.cut_score, al.next_score)):
        assert (np.isnan(g) and np.isnan(w)) or np.float32(g) == np.float32(w)


@pytest.mark.parametrize("mode", ["energy_ratio", "half_sigma2", "per_param"])
def test_weighted_allocation_bit_identical(ctx, mode):
    """UniRank's aggregated key I_l sigma^2 / ||Sigma_l||^2 (and weighted forms of the other
    keys) through score_and_allocate_weighted: bit-identical ranks, cut and used."""
    r = np.random.default_rng({"energy_ratio": 1, "half_sigma2": 2, "per_param": 3}[mode])
    sig, costs = [], []
    for u in range(40):
        m, n = int(r.integers(8, 600)), int(r.integers(8, 600))
        sig.append(np.sort(r.gamma(1.0, 1.0, size=min(m, n)))[::-1].astype(np.float32))
        costs.append(m + n)
    w = r.uniform(0.0, 2.0, len(sig)).astype(np.float32)
    w[3] = 0.0
    budget = int(0.35 * sum(len(s) * c for s, c in zip(sig, costs)))
    kmode = {"energy_ratio": K().KF_KEY_ENERGY_RATIO, "half_sigma2": K().KF_KEY_HALF_SIGMA2,
             "per_param": K().KF_KEY_PER_PARAM}[mode]
    sd = torch.from_numpy(np.concatenate(sig)).cuda()
    off = torch.tensor([0] + list(np.cumsum([len(s) for s in sig])), dtype=torch.int64, device="cuda")
    cost = torch.tensor(costs, dtype=torch.int64, device="cuda")
    ranks = torch.empty(len(sig), dtype=torch.int32, device="cuda")
    cut = torch.empty(2, dtype=torch.float32, device="cuda")
    used = torch.zeros(1, dtype=torch.int64, device="cuda")
    K().score_and_allocate_weighted(ctx, sd, off, cost, budget, ranks, mode=kmode, unit_weight=torch.from_numpy(w).cuda(),
                                    cut=cut, used=used)
    ctx.sync_status()
    al = O.allocate(sig, costs, budget, mode, precision="f32", weights=list(w))
    np.testing.assert_array_equal(ranks.cpu().numpy(), al.ranks)
    assert int(used.item()) == al.used
    c = cut.cpu().numpy()
    assert np.float32(c[0]) == np.float32(al.cut_score) and np.float32(c[1]) == np.float32(al.next_score)
    assert int(ranks[3].item()) == 0


def test_allocation_fixed_rank(ctx):
    ranks, cut, used = _gpu_alloc(ctx, [np.ones(5, np.float32), np.ones(3, np.float32)], [10, 20], 0,
                                  K().KF_FIXED_RANK, fixed=[4, 4])
    assert list(ranks) == [4, 3] and used == 4 * 10 + 3 * 20 and np.all(np.isnan(cut))


# ---------------------------------------------------------------- step 5b
@pytest.mark.parametrize("m,n,r", [(320, 192, 50), (192, 320, 77), (300, 300, 1), (257, 130, 130)])
def test_unwhiten(ctx, m, n, r):
    X, G, W = _factors(m, n, seed=m + n + r)
    oSx, oSg = O.cholesky_factors(X.astype(np.float64), G.astype(np.float64))
    Sx, Sg, Si, Wt = _gpu_whiten(ctx, X, G, W)
    s = min(m, n)
    sig = torch.empty(s, device="cuda")
    vec = torch.empty((s, s), device="cuda")
    K().whitened_svd(ctx, [Wt], [sig], [vec])
    U = torch.empty((m, r), device="cuda")
    V = torch.empty((r, n), device="cuda")
    K().unwhiten(ctx, bf16_dev(W, torch), Sx, Sg, Si, sig, vec, r, U, V)
    ctx.sync_status()
    Ut, so, Vt = O.whitened_svd(O.whiten(W, oSx, oSg))
    e_opt = float(np.sum(so[r:] ** 2))
    e = O.whitened_error(W, U.cpu().numpy(), V.cpu().numpy(), oSx, oSg)
    total = float(np.sum(so ** 2))
    if e_opt <= 1e-12 * total:
        assert e <= 1e-6 * total
    else:
        assert abs(e / e_opt - 1.0) <= 1e-3


# ---------------------------------------------------------------- end to end
def _run_pipeline(ctx, wl, streamed=False, chunk=256):
    from synth import device
    from vlm_compression_fac_b300 import pipeline
    units = pipeline.unit_specs(wl)
    weights = device.weights_on_device(wl, torch)
    quant = wl.quant == "int8_token"
    if not streamed:
        acts = {n: device.stream_on_device(wl, s, 0, wl.n_tokens, torch) for n, s in wl.sites.items() if s.kind == "act"}
        grads = {n: device.stream_on_device(wl, s, 0, wl.n_tokens, torch) for n, s in wl.sites.items() if s.kind == "grad"}
        res = pipeline.compress(ctx, units, weights, acts, grads, wl.n_tokens, lam=wl.lam, budget=wl.budget,
                                fixed_rank=wl.fixed_rank, quant=quant)
    else:
        blocks = sorted({u.block for u in wl.units})
        groups = [[i for i, u in enumerate(wl.units) if u.block == b] for b in blocks]
        res = pipeline.compress(ctx, units, weights, device.rows_fn(wl, torch), None, wl.n_tokens, lam=wl.lam,
                                budget=wl.budget, fixed_rank=wl.fixed_rank, quant=quant,
                                site_dims={n: s.d for n, s in wl.sites.items()},
                                act_sites=[n for n, s in wl.sites.items() if s.kind == "act"],
                                groups=groups, chunk_tokens=chunk)
    ctx.sync_status()
    return res


E2E = {
    "single_linear": (lambda: recipes.single_linear(), False),
    "mini_block": (lambda: recipes.mini_block(n_tokens=1200), False),
    "mini_block_qaw": (lambda: recipes.mini_block(n_tokens=1200, quant="int8_token", seed=91), False),
    "mini_model_streamed": (lambda: recipes.decoder_blocks(2, 256, 328, 128, 900, 0.4, 93, "mini_model"), True),
    "mini_vlm_heads_qaw_streamed": (lambda: recipes.mini_vlm(n_tokens=700), True),
}


@pytest.mark.parametrize("which", list(E2E))
def test_end_to_end(ctx, which):
    make, streamed = E2E[which]
    wl = make()
    res = _run_pipeline(ctx, wl, streamed=streamed)
    ref = O.compress_workload(wl)
    for name, cov in res.covs.items():
        assert rel_fro(cov.cpu().numpy(), ref["covs"][name]) <= 1e-4, name
    sig_o = [u.sigma for u in ref["units"]]
    for g, o in zip(res.units, ref["units"]):
        s_g = g.sigma.cpu().numpy()
        assert np.max(np.abs(s_g - o.sigma)) <= 1e-3 * o.sigma[0], g.name
    ranks = res.ranks.cpu().numpy()
    ok, moved = rank_parity(ranks, ref["alloc"], sig_o, 1e-6)
    assert ok, (ranks, ref["alloc"].ranks, moved)
    for g, o, u in zip(res.units, ref["units"], wl.units):
        r = g.rank
        e = O.whitened_error(recipes.gen_weight(wl, u), g.U.cpu().numpy(), g.V.cpu().numpy(), o.Sx, o.Sg)
        e_opt = float(np.sum(o.sigma[r:] ** 2))
        total = float(np.sum(o.sigma ** 2))
        if e_opt <= 1e-12 * total:
            assert e <= 1e-6 * total
        else:
            assert abs(e / e_opt - 1.0) <= 1e-3, (g.name, e, e_opt)
