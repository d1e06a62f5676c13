"""Parity at the full size of the Llama-7B-block workload (q, k, v, o 4096x4096; gate, up
4096x11008; down 11008x4096; N = 131072 bf16 tokens per site; 50% of the parameters kept),
run through pipeline.compress exactly as bench.py times it.

The oracle cannot regenerate 17 GB of calibration rows on the host in reasonable time, so:
  * covariances: sampled entries, each summed by the oracle over all N tokens from the
    generator's two columns (relative error of the entry <= 1e-4 of its scale), plus the
    damping identity X_ii - S_ii/N = lambda * mean(diag X) / (1 + lambda) on the GPU output;
  * steps 2-5: the oracle takes the GPU's finalised float32 X and G as its inputs (step
    parity) and computes in float64 the factors, W~ = S_x W S_g, the spectrum (Gram route,
    eigh) of every unit, the global allocation and the whitened error of the GPU's U V.
Tolerances are those of the small-shape parity tests (see test_gpu_parity.py).
"""
import numpy as np
import pytest

import oracle as O
from synth import recipes
from tests.gpu_util import host_weight, rank_parity, rel_fro

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def run():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from synth import device
    from vlm_compression_fac_b300 import kfsvd as K, pipeline
    wl = recipes.llama7b_block()
    ctx = K.Context(0)
    units = [pipeline.UnitSpec(u.name, u.m, u.n, u.x_site, u.g_site) for u in wl.units]
    acts = {n: device.stream_on_device(wl, s, 0, wl.n_tokens, torch) for n, s in wl.sites.items() if s.kind == "act"}
    grads = {n: device.stream_on_device(wl, s, 0, wl.n_tokens, torch) for n, s in wl.sites.items() if s.kind == "grad"}
    weights = {u.name: device.weight_on_device(wl, u, torch) for u in wl.units}
    res = pipeline.compress(ctx, units, weights, acts, grads, wl.n_tokens, lam=wl.lam, budget=wl.budget)
    ctx.sync_status()
    del acts, grads, weights
    covs = {k: v.cpu().numpy() for k, v in res.covs.items()}
    out = []
    for u in res.units:
        out.append(dict(name=u.name, m=u.m, n=u.n, sigma=u.sigma.cpu().numpy(), rank=u.rank,
                        U=u.U.cpu().numpy(), V=u.V.cpu().numpy(), Wt=u.Wt.cpu().numpy(), sweeps=u.sweeps))
    ranks = res.ranks.cpu().numpy()
    ctx.close()
    torch.cuda.empty_cache()
    return wl, covs, out, ranks


def _entry_sum(wl, site, i, j, chunk=32768):
    s = 0.0
    for t0 in range(0, wl.n_tokens, chunk):
        A = recipes.gen_stream(wl, site, t0, min(wl.n_tokens, t0 + chunk), cols=[i, j]).astype(np.float64)
        s += float(A[:, 0] @ A[:, 1])
    return s


@pytest.mark.parametrize("site_name", ["attn_in", "down_in", "gate_out", "k_out"])
def test_fullsize_covariance_sampled_entries(run, site_name):
    wl, covs, _, _ = run
    site = wl.sites[site_name]
    X = covs[site_name].astype(np.float64)
    d, N, lam = site.d, wl.n_tokens, wl.lam
    r = np.random.default_rng(d)
    out = list(recipes.outlier_channels(wl, site)[:2]) if site.kind == "act" else []
    pairs = [(0, 0), (d - 1, 0), (d - 1, d - 1)] + [(int(a), int(b)) for a, b in r.integers(0, d, (5, 2))]
    pairs += [(o, o) for o in out] + [(o, int(r.integers(0, d))) for o in out]
    diag_sum = {}
    for i, j in pairs:
        S_ij = _entry_sum(wl, site, i, j)
        if i == j:
            diag_sum[i] = S_ij
            continue
        S_ii = diag_sum.get(i) or _entry_sum(wl, site, i, i)
        S_jj = diag_sum.get(j) or _entry_sum(wl, site, j, j)
        diag_sum[i], diag_sum[j] = S_ii, S_jj
        scale = np.sqrt(S_ii * S_jj) / N
        assert abs(X[i, j] - S_ij / N) <= 1e-4 * scale, (site_name, i, j)
        assert X[i, j] == X[j, i]
    # damping: every diagonal entry carries the same lambda * mean(diag X) / (1 + lambda)
    delta = lam * float(np.mean(np.diag(X))) / (1.0 + lam)
    for i, S_ii in diag_sum.items():
        assert abs((X[i, i] - S_ii / N) - delta) <= 1e-4 * (S_ii / N + delta), (site_name, i)


def test_fullsize_spectra_allocation_and_factors(run):
    wl, covs, out, ranks = run
    sig_o, whitened = [], []
    for u, g in zip(wl.units, out):
        X = covs[u.x_site].astype(np.float64)
        G = covs[u.g_site].astype(np.float64)
        Sx, Sg = O.cholesky_factors(X, G)
        W = host_weight(wl, u, torch).astype(np.float64)
        Wt = O.whiten(W, Sx, Sg)
        assert rel_fro(g["Wt"], Wt) <= 1e-5, u.name
        lam_ = O.gram_eigenvalues(Wt)
        so = np.sqrt(np.maximum(lam_, 0.0))
        sig_o.append(so)
        assert np.all(np.diff(g["sigma"]) <= 0), u.name
        assert np.max(np.abs(g["sigma"] - so)) <= 1e-3 * so[0], u.name
        assert 1 <= g["sweeps"] <= 30
        whitened.append((W, Sx, Sg))
    costs = [u.m + u.n for u in wl.units]
    problems = []
    # ranks: the oracle's allocation fed the GPU's float32 spectra is bit-identical ...
    al32 = O.allocate([g["sigma"] for g in out], costs, wl.budget, precision="f32")
    np.testing.assert_array_equal(ranks, al32.ranks)
    # ... and against the oracle's own spectra they differ at most at score ties near the cut
    al = O.allocate(sig_o, costs, wl.budget)
    ok, moved = rank_parity(ranks, al, sig_o, 1e-6)
    sig_err = max(float(np.max(np.abs(g["sigma"] / so - 1.0)[:g["rank"] + 8])) for g, so in zip(out, sig_o))
    if not ok:
        problems.append(("ranks", list(ranks), list(al.ranks), moved,
                         "max rel sigma error over the kept components %.3g" % sig_err))
    assert int(np.sum(ranks * np.asarray(costs))) <= wl.budget
    # whitened error of the GPU factors against the optimum at the same rank
    for (W, Sx, Sg), g, so in zip(whitened, out, sig_o):
        r = g["rank"]
        assert g["U"].shape == (g["m"], r) and g["V"].shape == (r, g["n"])
        e = O.whitened_error(W, g["U"], g["V"], Sx, Sg)
        e_opt = float(np.sum(so[r:] ** 2))
        if abs(e / e_opt - 1.0) > 1e-3:
            problems.append(("whitened error", g["name"], e, e_opt))
    assert not problems, problems
