"""The Python glue of the pipeline drivers, on CPU: every libkfsvd call is replaced for the
test by a stand-in built from the fp64 oracle (tests/cpu_abi_standin.py), so what is checked
is the bookkeeping around the calls (unit order, factor sharing, index sets, the budget and
the dense cost, which factors are mapped back), against the oracle's own whole-workload
flows.  The kernels themselves are checked on the GPU by the gpu-marked tests."""
import numpy as np
import pytest
import torch

import oracle as O
from synth import recipes
from tests import cpu_abi_standin as standin


def _inputs(wl):
    from vlm_compression_fac_b300 import pipeline
    units = pipeline.unit_specs(wl)
    weights = {}
    for u in wl.units:
        weights.setdefault(u.weight, torch.from_numpy(recipes.gen_full_weight(wl, u)))
    acts = {n: torch.from_numpy(recipes.gen_stream(wl, s, 0, wl.n_tokens)) for n, s in wl.sites.items()
            if s.kind == "act"}
    grads = {n: torch.from_numpy(recipes.gen_stream(wl, s, 0, wl.n_tokens)) for n, s in wl.sites.items()
             if s.kind == "grad"}
    return units, weights, acts, grads


def _small():
    return recipes.mini_block(n_tokens=300, d=64, ffn=96, kv=32, seed=5)


@pytest.mark.parametrize("heads", [False, True])
def test_compress_glue(monkeypatch, heads):
    from vlm_compression_fac_b300 import pipeline
    ctx = standin.install(monkeypatch)
    wl = recipes.mini_vlm(n_tokens=200) if heads else _small()
    units, weights, acts, grads = _inputs(wl)
    res = pipeline.compress(ctx, units, weights, acts, grads, wl.n_tokens, lam=wl.lam, budget=wl.budget,
                            quant=wl.quant == "int8_token")
    ref = O.compress_workload(wl)
    sig = [u.sigma.numpy() for u in res.units]
    for s_, r in zip(sig, ref["units"]):
        np.testing.assert_allclose(s_, r.sigma, rtol=1e-5, atol=1e-7 * r.sigma[0])
    al = O.allocate(sig, [u.m + u.n for u in wl.units], wl.budget, precision="f32")
    np.testing.assert_array_equal(res.ranks.numpy(), al.ranks)
    for g, r, u in zip(res.units, ref["units"], wl.units):
        e = O.whitened_error(recipes.gen_weight(wl, u), g.U.numpy(), g.V.numpy(), r.Sx, r.Sg)
        opt = float(np.sum(r.sigma[g.rank:] ** 2))
        assert abs(e - opt) <= 1e-4 * max(opt, 1e-6 * float(np.sum(r.sigma ** 2))), u.name


def test_hybrid_glue_matches_the_oracle_flow(monkeypatch):
    from vlm_compression_fac_b300 import pipeline
    ctx = standin.install(monkeypatch)
    wl = _small()
    units, weights, acts, grads = _inputs(wl)
    names = [u.name for u in wl.units]
    pair = (names.index("gate"), names.index("up"))
    res = pipeline.compress_hybrid_ffn(ctx, units, weights, acts, grads, wl.n_tokens, wl.lam, wl.budget,
                                       r_temp=8, n_svd=40, pairs=[pair])
    ref = O.compress_hybrid_ffn(wl, r_temp=8, n_svd=40, pairs=[pair])
    np.testing.assert_array_equal(res.splits[0]["svd"].numpy(), ref["splits"][0]["svd"])
    np.testing.assert_array_equal(res.splits[0]["dense"].numpy(), ref["splits"][0]["dense"])
    assert res.dense_cost == ref["dense_cost"] and res.budget == ref["budget"]
    assert [(e.kind, e.unit) for e in res.entries] == [(k, i) for k, i, _ in ref["entries"]]
    for e, (_, _, r) in zip(res.entries, ref["entries"]):
        np.testing.assert_allclose(e.out.sigma.numpy(), r.sigma, rtol=1e-5, atol=1e-7 * r.sigma[0])
    sig = [e.out.sigma.numpy() for e in res.entries]
    al = O.allocate(sig, [e.out.m + e.out.n for e in res.entries], ref["budget"], precision="f32")
    np.testing.assert_array_equal(res.ranks.numpy(), al.ranks)
    assert int(res.used.item()) == al.used <= res.budget
    # the SVD-branch factors reproduce the selected columns' optimum
    for e, (_, _, r) in zip(res.entries, ref["entries"]):
        if e.kind != "svd":
            continue
        W = recipes.gen_weight(wl, wl.units[e.unit])[:, e.svd_idx.numpy()]
        err = O.whitened_error(W, e.out.U.numpy(), e.out.V.numpy(), r.Sx, r.Sg)
        opt = float(np.sum(r.sigma[e.out.rank:] ** 2))
        assert abs(err - opt) <= 1e-4 * max(opt, 1e-6 * float(np.sum(r.sigma ** 2)))


def test_fisher_and_activation_only_glue(monkeypatch):
    from vlm_compression_fac_b300 import pipeline
    ctx = standin.install(monkeypatch)
    wl = _small()
    units, weights, acts, grads = _inputs(wl)
    res = pipeline.compress(ctx, units, weights, acts, grads, wl.n_tokens, lam=wl.lam, budget=wl.budget,
                            score="empirical_fisher")
    keys = [g.scores.numpy() for g in res.units]
    al = O.allocate_keys(keys, [u.m + u.n for u in wl.units], wl.budget)
    np.testing.assert_array_equal(res.ranks.numpy(), al.ranks)
    n_keep = int(al.ranks.sum())
    for ui, g in enumerate(res.units):
        want = np.sort(al.order_comp[:n_keep][al.order_unit[:n_keep] == ui])
        np.testing.assert_array_equal(g.kept.numpy(), want)
        assert g.U.shape == (g.m, len(want)) and g.V.shape == (len(want), g.n)
    act = pipeline.compress_activation_only(ctx, units, weights, acts, wl.n_tokens, wl.budget)
    ref = O.compress_workload_activation_only(wl)
    np.testing.assert_array_equal(act.ranks.numpy(), ref["alloc"].ranks)
    for g, r in zip(act.units, ref["units"]):
        np.testing.assert_allclose(g.U.numpy() @ g.V.numpy(), r["U"] @ r["Vt"], atol=1e-5)


def test_units_larger_than_dense_are_reported(monkeypatch):
    """A generous budget lets the allocation keep more than a unit's dense size,
    r (m + n) > m n; the result names those units."""
    from vlm_compression_fac_b300 import pipeline
    ctx = standin.install(monkeypatch)
    wl = _small()
    units, weights, acts, grads = _inputs(wl)
    total = sum(u.m * u.n for u in wl.units)
    res = pipeline.compress(ctx, units, weights, acts, grads, wl.n_tokens, lam=wl.lam, budget=2 * total)
    big = res.larger_than_dense()
    want = [u.name for u, r in zip(wl.units, res.ranks.tolist()) if r * (u.m + u.n) > u.m * u.n]
    assert big == want and len(big) > 0
    res = pipeline.compress(ctx, units, weights, acts, grads, wl.n_tokens, lam=wl.lam, budget=wl.budget // 4)
    assert res.larger_than_dense() == []


@pytest.mark.parametrize("score", [None, "empirical_fisher"])
def test_streamed_groups_match_resident_rows(monkeypatch, score):
    """Rows produced on demand in uneven token chunks, units processed block by block with the
    covariances released after each block, quantised activation sites: the same spectra,
    ranks and factors as with every site's rows resident and one group."""
    from vlm_compression_fac_b300 import pipeline
    ctx = standin.install(monkeypatch)
    wl = recipes.decoder_blocks(2, 64, 96, 32, 250, 0.4, 17, "two_blocks", quant="int8_token")
    units, weights, acts, grads = _inputs(wl)
    one = pipeline.compress(ctx, units, weights, acts, grads, wl.n_tokens, lam=wl.lam, budget=wl.budget,
                            quant=True, score=score)

    def rows(name, t0, t1):
        return torch.from_numpy(recipes.gen_stream(wl, wl.sites[name], t0, t1))

    blocks = sorted({u.block for u in wl.units})
    groups = [[i for i, u in enumerate(wl.units) if u.block == b] for b in blocks]
    streamed = pipeline.compress(ctx, units, weights, rows, None, wl.n_tokens, lam=wl.lam, budget=wl.budget,
                                 quant=True, score=score, site_dims={n: s.d for n, s in wl.sites.items()},
                                 act_sites=[n for n, s in wl.sites.items() if s.kind == "act"], groups=groups,
                                 chunk_tokens=97, keep_covs=False, keep_whitened=False)
    # the covariances are held in float32 between chunks (as in the library), so chunking moves
    # the sums by float32 roundings: compare against sigma_max and max |U V|
    assert streamed.ranks.tolist() == one.ranks.tolist()
    for a, b in zip(streamed.units, one.units):
        sb = b.sigma.numpy()
        np.testing.assert_allclose(a.sigma.numpy(), sb, rtol=0, atol=1e-5 * sb[0])
        pb = (b.U @ b.V).numpy()
        np.testing.assert_allclose((a.U @ a.V).numpy(), pb, rtol=0, atol=1e-4 * np.abs(pb).max())
    assert streamed.covs == {}
