"""Swift-SVD's activation-only route on the GPU against the fp64 oracle: the output
covariance C = W^T X W, its eigenpairs, the factors W V_k / V_k^T, and the whole route over
small workloads (ragged shapes, several tiles, attention heads with INT8 fake-quantised
activations).

Tolerances: C relative Frobenius <= 1e-5 (float32 operands as three bf16 planes); sigma
within 1e-3 sigma_max (the contract's spectrum tolerance); the activation-aware loss of the
GPU's factors within 1e-3 (relative) of the optimum, the sum of the dropped eigenvalues, or
1e-6 of the total where that optimum is ~0; the oracle's allocation fed the GPU's float32
spectra gives bit-identical ranks.
"""
import numpy as np
import pytest

import oracle as O
from synth import recipes
from tests.gpu_util import bf16_dev, rel_fro, to_dev

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


def _rows(rng, N, m):
    A = rng.standard_normal((N, m)) * np.exp(rng.standard_normal(m))[None, :]
    return recipes.philox.bf16_bits_to_f32(recipes.philox.f32_to_bf16_bits(A.astype(np.float32)))


@pytest.mark.parametrize("m,n,wdt", [(320, 192, "bf16"), (200, 328, "f32"), (130, 130, "bf16")])
def test_output_covariance(ctx, m, n, wdt):
    rng = np.random.default_rng(m + n)
    A = _rows(rng, 900, m)
    X = O.finalize_covariance(O.covariance_sum(A), len(A), 0.0).astype(np.float32)
    W = (rng.standard_normal((m, n)) * 0.02).astype(np.float32)
    if wdt == "bf16":
        W = recipes.philox.bf16_bits_to_f32(recipes.philox.f32_to_bf16_bits(W))
        Wd = bf16_dev(W, torch)
    else:
        Wd = to_dev(W, torch)
    C = torch.empty((n, n), device="cuda")
    K().activation_covariance(ctx, to_dev(X, torch), Wd, C)
    ctx.sync_status()
    want = W.astype(np.float64).T @ X.astype(np.float64) @ W.astype(np.float64)
    assert rel_fro(C.cpu().numpy(), want) <= 1e-5


@pytest.mark.parametrize("n,nprob", [(192, 2), (328, 1), (64, 3), (1, 1)])
def test_eigenpairs_and_factors(ctx, n, nprob):
    rng = np.random.default_rng(n * 7 + nprob)
    m = n + 37
    Cs, As, Ws = [], [], []
    for _ in range(nprob):
        A = _rows(rng, 700, m)
        W = (rng.standard_normal((m, n)) * 0.02).astype(np.float32)
        Cs.append(O.output_covariance(A, W).astype(np.float32))
        As.append(A)
        Ws.append(W)
    sig = [torch.empty(n, device="cuda") for _ in range(nprob)]
    vec = [torch.empty((n, n), device="cuda") for _ in range(nprob)]
    sw = torch.zeros(nprob, dtype=torch.int32, device="cuda")
    K().activation_eig(ctx, [to_dev(C, torch) for C in Cs], sig, vec, sweeps=sw)
    ctx.sync_status()
    for i in range(nprob):
        so, _ = O.output_eig(Cs[i].astype(np.float64))
        sg = sig[i].cpu().numpy()
        assert np.all(np.diff(sg) <= 0)
        assert np.max(np.abs(sg - so)) <= 1e-3 * so[0]
        V = vec[i].cpu().numpy().astype(np.float64)
        np.testing.assert_allclose(V.T @ V, np.eye(n), atol=1e-4)
        for k in sorted({0, 1, n // 3, n // 2, n}):
            U = torch.empty((m, max(k, 1)), device="cuda")[:, :k]
            Vt = torch.empty((max(k, 1), n), device="cuda")[:k]
            K().activation_factors(ctx, to_dev(Ws[i], torch), vec[i], k, U, Vt)
            ctx.sync_status()
            Uh, Vh = U.cpu().numpy(), Vt.cpu().numpy()
            np.testing.assert_array_equal(Vh, V[:, :k].T.astype(np.float32))
            if k:
                assert rel_fro(Uh, Ws[i].astype(np.float64) @ V[:, :k]) <= 1e-4
            loss = O.activation_loss(As[i], Ws[i], Uh, Vh)
            opt = float(np.sum(so[k:] ** 2))
            tot = float(np.sum(so ** 2))
            assert abs(loss - opt) <= 1e-3 * max(opt, 1e-3 * tot), (k, loss, opt)


@pytest.mark.parametrize("name", ["mini_block", "mini_vlm_heads_qaw"])
def test_end_to_end_activation_only(ctx, name):
    from synth import device
    from vlm_compression_fac_b300 import pipeline
    wl = recipes.mini_block(n_tokens=1000, seed=97) if name == "mini_block" else recipes.mini_vlm(n_tokens=700)
    units = pipeline.unit_specs(wl)
    weights = device.weights_on_device(wl, torch)
    acts = {n: device.stream_on_device(wl, s, 0, wl.n_tokens, torch) for n, s in wl.sites.items() if s.kind == "act"}
    res = pipeline.compress_activation_only(ctx, units, weights, acts, wl.n_tokens, wl.budget,
                                            quant=wl.quant == "int8_token")
    ctx.sync_status()
    ref = O.compress_workload_activation_only(wl)
    sig_g = [g.sigma.cpu().numpy() for g in res.units]
    for g, r, sg in zip(res.units, ref["units"], sig_g):
        assert np.max(np.abs(sg - r["sigma"])) <= 1e-3 * r["sigma"][0], g.name
    costs = [u.m + u.n for u in wl.units]
    al = O.allocate([s[:min(u.m, u.n)] for s, u in zip(sig_g, wl.units)], costs, wl.budget, precision="f32")
    np.testing.assert_array_equal(res.ranks.cpu().numpy(), al.ranks)
    assert int(res.used.item()) == al.used <= wl.budget
    # ranks against the oracle's own: differences only at ties within 1e-6 of the cut
    cut = ref["alloc"].cut_score
    for g, r in zip(res.units, ref["units"]):
        if g.rank != r["rank"]:
            lo, hi = sorted((g.rank, r["rank"]))
            sc = 0.5 * r["sigma"][lo:hi] ** 2
            assert np.all(np.abs(sc - cut) <= 1e-6 * abs(cut)), (g.name, g.rank, r["rank"])
    for g, r, u in zip(res.units, ref["units"], wl.units):
        A = recipes.gen_stream(wl, wl.sites[u.x_site], 0, wl.n_tokens)
        if wl.quant == "int8_token":
            A = O.fake_quant_int8_token(A)
        A = A[:, u.x_off:u.x_off + u.m]
        loss = O.activation_loss(A, r["W"], g.U.cpu().numpy(), g.V.cpu().numpy())
        opt = float(np.sum(r["sigma"][g.rank:] ** 2))
        tot = float(np.sum(r["sigma"] ** 2))
        assert abs(loss - opt) <= 1e-3 * max(opt, 1e-3 * tot), (g.name, loss, opt)


def test_llama7b_block_activation_only_fullsize(ctx):
    """The route over the Llama-7B-shaped block at full size (N = 131072; q, k, v, o 4096^2,
    gate/up 4096 x 11008 whose output covariances are 11008^2, down 11008 x 4096), with the
    checks the oracle can afford: sampled entries of q's C against float64 sums over all
    tokens; sigma against a float64 eigendecomposition of the GPU's own C (q, down); for the
    11008^2 problems, eigen-residual bounds |lambda_i - lambda(C)| <= ||C v_i - lambda_i v_i||;
    the loss of the kept subspace, tr((I - P) C (I - P)), against the optimum; allocation
    bit-identical on the GPU's spectra."""
    import time
    from synth import device
    from vlm_compression_fac_b300 import pipeline
    wl = recipes.llama7b_block()
    units = pipeline.unit_specs(wl)
    weights = device.weights_on_device(wl, torch)
    acts = {n: device.stream_on_device(wl, s, 0, wl.n_tokens, torch) for n, s in wl.sites.items() if s.kind == "act"}
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    res = pipeline.compress_activation_only(ctx, units, weights, acts, wl.n_tokens, wl.budget, keep_cov=True)
    ctx.sync_status()
    print("llama7b_block activation-only route: %.2f s, sweeps %s, ranks %s" % (
        time.perf_counter() - t0, [g.sweeps for g in res.units], res.ranks.cpu().tolist()))
    sig_g = [g.sigma.cpu().numpy() for g in res.units]
    costs = [u.m + u.n for u in wl.units]
    al = O.allocate([s[:min(u.m, u.n)] for s, u in zip(sig_g, wl.units)], costs, wl.budget, precision="f32")
    np.testing.assert_array_equal(res.ranks.cpu().numpy(), al.ranks)
    assert int(res.used.item()) == al.used <= wl.budget
    names = [u.name for u in wl.units]

    # sampled entries of q's output covariance against float64 sums over all tokens
    iq = names.index("q")
    Wq = recipes.gen_weight(wl, wl.units[iq]).astype(np.float64)
    cols = [0, 1, 2000, 4095, 77]
    Y = np.zeros((0, len(cols)))
    A_dev = acts[wl.units[iq].x_site]
    sums = np.zeros((len(cols), len(cols)))
    for t in range(0, wl.n_tokens, 16384):
        A = A_dev[t:t + 16384].float().cpu().numpy().astype(np.float64)
        Y = A @ Wq[:, cols]
        sums += Y.T @ Y
    Cq = res.units[iq].C.cpu().numpy().astype(np.float64)
    for a, b in [(0, 0), (1, 2), (3, 4), (0, 3)]:
        want = sums[a, b] / wl.n_tokens
        scale = np.sqrt(sums[a, a] * sums[b, b]) / wl.n_tokens
        assert abs(Cq[cols[a], cols[b]] - want) <= 1e-4 * scale, (cols[a], cols[b])

    for i, g in enumerate(res.units):
        C = g.C.cpu().numpy().astype(np.float64)
        C = 0.5 * (C + C.T)
        k = int(g.rank)
        V = g.vecs.cpu().numpy().astype(np.float64)[:, :k]
        CV = C @ V
        lam = sig_g[i].astype(np.float64)[:k] ** 2
        trC = float(np.trace(C))
        loss = trC - 2.0 * float(np.sum(V * CV)) + float(np.sum((V.T @ V) * (V.T @ CV)))
        if g.name in ("q", "down"):
            so = np.sqrt(np.maximum(np.linalg.eigvalsh(C)[::-1], 0.0))
            assert np.max(np.abs(sig_g[i] - so)) <= 1e-3 * so[0], g.name
            opt = float(np.sum(so[k:] ** 2))
        else:
            resid = np.linalg.norm(CV - V * lam[None, :], axis=0)
            assert np.all(resid <= 1e-3 * lam[0]), (g.name, float(resid.max() / lam[0]))
            opt = trC - float(np.sum(lam))
        assert abs(loss - opt) <= 1e-3 * max(opt, 1e-3 * trC), (g.name, loss, opt)


def test_activation_only_streamed_blocks(ctx):
    """The route with rows generated on demand in token chunks and the units processed block by
    block (two decoder blocks, INT8 fake-quantised activations): the same checks as the
    resident case against the oracle."""
    from synth import device
    from vlm_compression_fac_b300 import pipeline
    wl = recipes.decoder_blocks(2, 256, 328, 128, 900, 0.4, 31, "two_blocks_qaw", quant="int8_token")
    units = pipeline.unit_specs(wl)
    weights = device.weights_on_device(wl, torch)
    blocks = sorted({u.block for u in wl.units})
    groups = [[i for i, u in enumerate(wl.units) if u.block == b] for b in blocks]
    res = pipeline.compress_activation_only(ctx, units, weights, device.rows_fn(wl, torch), wl.n_tokens, wl.budget,
                                            quant=True, site_dims={n: s.d for n, s in wl.sites.items()},
                                            groups=groups, chunk_tokens=256)
    ctx.sync_status()
    ref = O.compress_workload_activation_only(wl)
    sig_g = [g.sigma.cpu().numpy() for g in res.units]
    for g, r, sg in zip(res.units, ref["units"], sig_g):
        assert np.max(np.abs(sg - r["sigma"])) <= 1e-3 * r["sigma"][0], g.name
    costs = [u.m + u.n for u in wl.units]
    al = O.allocate([s[:min(u.m, u.n)] for s, u in zip(sig_g, wl.units)], costs, wl.budget, precision="f32")
    np.testing.assert_array_equal(res.ranks.cpu().numpy(), al.ranks)
    for g, r, u in zip(res.units, ref["units"], wl.units):
        A = O.fake_quant_int8_token(recipes.gen_stream(wl, wl.sites[u.x_site], 0, wl.n_tokens))
        loss = O.activation_loss(A[:, u.x_off:u.x_off + u.m], r["W"], g.U.cpu().numpy(), g.V.cpu().numpy())
        opt = float(np.sum(r["sigma"][g.rank:] ** 2))
        tot = float(np.sum(r["sigma"] ** 2))
        assert abs(loss - opt) <= 1e-3 * max(opt, 1e-3 * tot), (g.name, loss, opt)
