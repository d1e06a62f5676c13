"""LASER's hybrid FFN channel selection on the GPU against the fp64 oracle, and the index
plumbing it uses (ordered mask compaction, row/column gathers: bit-exact).

Tolerances: a channel error is e_j = d_j^T X d_j with d_j = (W - U V)[:, j]; U V is formed
from three-plane bf16 operands, i.e. to float32 precision, so d_j carries an absolute error
of about eps32 |w_j| however small d_j is (the cancellation when U V ~ W), and
|de_j| <= 2 sqrt(e_j) sqrt(dd^T X dd) ~ 2 eps32 sqrt(e_j w_j^T X w_j).  The tests allow
1e-4 e_j + 2e-6 sqrt(e_j w_j^T X w_j) (about 17 eps32) against the oracle's float64 error of
the same inputs; the split fed the GPU's float32 keys is identical to the oracle's split of
those keys; against the oracle's own temporary SVD the errors agree within 1e-3 of the largest.
"""
import numpy as np
import pytest

import oracle as O
from synth import recipes
from tests.gpu_util import bf16_dev, to_dev

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


@pytest.mark.parametrize("n", [0, 1, 1023, 1024, 5000])
def test_compact_mask_and_gather(ctx, n):
    rng = np.random.default_rng(n + 3)
    mask = (rng.random(n) < 0.37).astype(np.uint8)
    md = torch.from_numpy(mask).cuda() if n else torch.empty(0, dtype=torch.uint8, device="cuda")
    for want in (0, 1):
        idx = K().compact_mask(ctx, md, want)
        ctx.sync_status()
        np.testing.assert_array_equal(idx.cpu().numpy(), np.nonzero((mask != 0) == bool(want))[0])
    src = rng.standard_normal((37, max(n, 1) + 5)).astype(np.float32)
    cols = np.nonzero(mask)[0]
    rows = rng.integers(0, 37, 11)
    for dt in ("f32", "bf16"):
        s_h = src if dt == "f32" else recipes.philox.bf16_bits_to_f32(recipes.philox.f32_to_bf16_bits(src))
        s_d = to_dev(s_h, torch) if dt == "f32" else bf16_dev(s_h, torch)
        ci = torch.from_numpy(cols).cuda()
        ri = torch.from_numpy(rows.astype(np.int64)).cuda()
        g = K().gather_rows_cols(ctx, s_d, row_idx=ri, col_idx=ci)
        ctx.sync_status()
        np.testing.assert_array_equal(g.float().cpu().numpy(), s_h[rows][:, cols])
        g = K().gather_rows_cols(ctx, s_d, col_idx=ci)
        ctx.sync_status()
        np.testing.assert_array_equal(g.float().cpu().numpy(), s_h[:, cols])


@pytest.mark.parametrize("m,n,r,wdt", [(320, 704, 64, "bf16"), (130, 257, 0, "f32"), (200, 96, 96, "bf16")])
def test_channel_errors(ctx, m, n, r, wdt):
    rng = np.random.default_rng(m + n + r)
    A = rng.standard_normal((600, m)).astype(np.float32)
    X = O.finalize_covariance(O.covariance_sum(A), 600, 1e-2).astype(np.float32)
    W = (rng.standard_normal((m, n)) * 0.02).astype(np.float32)
    if wdt == "bf16":
        W = recipes.philox.bf16_bits_to_f32(recipes.philox.f32_to_bf16_bits(W))
        Wd = bf16_dev(W, torch)
    else:
        Wd = to_dev(W, torch)
    if r:
        # the rank-r truncation of W plus a little noise: small, uneven per-channel errors
        u, s, vt = np.linalg.svd(W.astype(np.float64), full_matrices=False)
        U = (u[:, :r] * s[:r]).astype(np.float32)
        V = (vt[:r] + 1e-4 * rng.standard_normal((r, n))).astype(np.float32)
        Ud, Vd = to_dev(U, torch), to_dev(V, torch)
    else:
        U = np.zeros((m, 0), np.float32)
        V = np.zeros((0, n), np.float32)
        Ud = Vd = None
    err = torch.zeros(n, dtype=torch.float64, device="cuda")
    keys = torch.empty(n, dtype=torch.float32, device="cuda")
    K().channel_errors(ctx, Wd, Ud, Vd, to_dev(X, torch), err, keys=keys)
    ctx.sync_status()
    want = O.channel_errors(W, U, V, X)
    dense = O.channel_errors(W, np.zeros((m, 0)), np.zeros((0, n)), X)   # w_j^T X w_j
    got = err.cpu().numpy()
    assert np.all(np.abs(got - want) <= 1e-4 * want + 2e-6 * np.sqrt(want * dense))
    np.testing.assert_array_equal(keys.cpu().numpy(), got.astype(np.float32))


def test_hybrid_split_on_a_block(ctx):
    from synth import device
    from vlm_compression_fac_b300 import pipeline
    wl = recipes.mini_block(n_tokens=1000, seed=98)
    units = pipeline.unit_specs(wl)
    weights = device.weights_on_device(wl, torch)
    acts = {n: device.stream_on_device(wl, s, 0, wl.n_tokens, torch) for n, s in wl.sites.items() if s.kind == "act"}
    grads = {n: device.stream_on_device(wl, s, 0, wl.n_tokens, torch) for n, s in wl.sites.items() if s.kind == "grad"}
    res = pipeline.compress(ctx, units, weights, acts, grads, wl.n_tokens, lam=wl.lam, budget=None,
                            defer_allocation=True, keep_covs=["mlp_in"])
    names = [u.name for u in wl.units]
    r_t, n_svd = 64, 400
    facs = {}
    for nm in ("gate", "up"):
        o = res.units[names.index(nm)]
        U = torch.empty((o.m, r_t), device="cuda")
        V = torch.empty((r_t, o.n), device="cuda")
        K().unwhiten(ctx, weights[nm], o.Sx, o.Sg, o.Sinv, o.sigma, o.vecs, r_t, U, V)
        facs[nm] = (U, V)
    X = res.covs["mlp_in"]
    svd, dense, err, keys = pipeline.hybrid_ffn_split(ctx, weights["gate"], weights["up"], X, facs["gate"],
                                                      facs["up"], n_svd)
    ctx.sync_status()
    f = wl.units[names.index("gate")].n
    assert len(svd) == n_svd and len(dense) == f - n_svd
    assert sorted(np.concatenate([svd.cpu().numpy(), dense.cpu().numpy()]).tolist()) == list(range(f))
    # the oracle's split of the GPU's float32 keys is the GPU's split
    np.testing.assert_array_equal(svd.cpu().numpy(), O.select_svd_channels([keys.cpu().numpy()], n_svd))
    # errors of the GPU's temporary factors, in float64
    Xh = X.cpu().numpy().astype(np.float64)
    Ws = {nm: recipes.gen_weight(wl, wl.units[names.index(nm)]) for nm in ("gate", "up")}
    want = sum(O.channel_errors(Ws[nm], facs[nm][0].cpu().numpy(), facs[nm][1].cpu().numpy(), Xh)
               for nm in ("gate", "up"))
    dense = sum(O.channel_errors(Ws[nm], np.zeros((Ws[nm].shape[0], 0)), np.zeros((0, f)), Xh)
                for nm in ("gate", "up"))
    got = err.cpu().numpy()
    assert np.all(np.abs(got - want) <= 1e-4 * want + 2e-6 * np.sqrt(want * dense))
    # against the oracle's own temporary SVD (its factors differ only by the eigensolver's error)
    ref = O.compress_workload(wl, units=[names.index("gate"), names.index("up")])
    Xo = ref["covs"]["mlp_in"]
    own = 0.0
    for ur, nm in zip(ref["units"], ("gate", "up")):
        Uo, Vo = O.unwhiten(ur.Sx, ur.Sg, ur.U_t, ur.sigma, ur.V_t, r_t)
        own = own + O.channel_errors(recipes.gen_weight(wl, wl.units[names.index(nm)]), Uo, Vo, Xo)
    assert np.max(np.abs(got - own)) <= 1e-3 * own.max()


def test_hybrid_flow_end_to_end(ctx):
    """The whole hybrid FFN flow on a block: the split fed the GPU's keys is the oracle's split
    of them; every entry's spectrum within 1e-3 sigma_max of the oracle's whitening of the same
    columns (its G block taken at the GPU's SVD-friendly set); the allocation over the entries,
    with the dense cost off the budget, bit-identical on the GPU's spectra; every entry's
    factors at the whitened optimum within 1e-3."""
    from synth import device
    from vlm_compression_fac_b300 import pipeline
    wl = recipes.mini_block(n_tokens=1000, seed=99)
    units = pipeline.unit_specs(wl)
    weights = device.weights_on_device(wl, torch)
    acts = {n: device.stream_on_device(wl, s, 0, wl.n_tokens, torch) for n, s in wl.sites.items() if s.kind == "act"}
    grads = {n: device.stream_on_device(wl, s, 0, wl.n_tokens, torch) for n, s in wl.sites.items() if s.kind == "grad"}
    names = [u.name for u in wl.units]
    gi, ui = names.index("gate"), names.index("up")
    res = pipeline.compress_hybrid_ffn(ctx, units, weights, acts, grads, wl.n_tokens, wl.lam, wl.budget,
                                       r_temp=64, n_svd=400, pairs=[(gi, ui)])
    ctx.sync_status()
    sp = res.splits[0]
    S = sp["svd"].cpu().numpy()
    np.testing.assert_array_equal(S, O.select_svd_channels([sp["keys"].cpu().numpy()], 400))
    f = wl.units[gi].n
    assert res.dense_cost == 2 * wl.units[gi].m * (f - 400) and res.budget == wl.budget - res.dense_cost
    ref = O.compress_workload(wl)
    sig = []
    for e in res.entries:
        r = ref["units"][e.unit]
        u = wl.units[e.unit]
        W = recipes.gen_weight(wl, u).astype(np.float64)
        if e.kind == "svd":
            W = W[:, S]
            Sx, Sg = O.cholesky_factors(r.X, r.G[np.ix_(S, S)])
        else:
            Sx, Sg = r.Sx, r.Sg
        so = np.sqrt(np.maximum(O.gram_eigenvalues(O.whiten(W, Sx, Sg)), 0.0))
        sg = e.out.sigma.cpu().numpy()
        assert np.max(np.abs(sg - so)) <= 1e-3 * so[0], (e.kind, u.name)
        sig.append(sg)
        k = int(e.out.rank)
        err = O.whitened_error(W, e.out.U.cpu().numpy(), e.out.V.cpu().numpy(), Sx, Sg)
        opt = float(np.sum(so[k:] ** 2))
        assert abs(err - opt) <= 1e-3 * max(opt, 1e-6 * float(np.sum(so ** 2))), (e.kind, u.name, err, opt)
    al = O.allocate(sig, [e.out.m + e.out.n for e in res.entries], res.budget, precision="f32")
    np.testing.assert_array_equal(res.ranks.cpu().numpy(), al.ranks)
    assert int(res.used.item()) == al.used <= res.budget
