"""Edge cases of every call on the GPU: empty inputs, one token, degenerate spectra (a zero
weight, a rank-one weight), vector-shaped layers (min(m, n) = 1), an empty allocation pool,
budgets of zero and of everything, full-rank and rank-zero factors."""
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


def test_accumulate_zero_and_one_token(ctx):
    wl = recipes.mini_block(n_tokens=8)
    A = recipes.gen_stream(wl, wl.sites["attn_in"], 0, 1)
    d = A.shape[1]
    cov = torch.full((d, d), 3.0, device="cuda")
    rows = bf16_dev(A, torch)
    K().kfac_accumulate(ctx, rows[:0], cov)          # no tokens: nothing changes
    ctx.sync_status()
    assert torch.all(cov == 3.0)
    cov.zero_()
    K().kfac_accumulate(ctx, rows[:1], cov)          # one token: the outer product, exactly
    ctx.sync_status()
    want = np.tril(np.outer(A[0], A[0]).astype(np.float32))
    np.testing.assert_array_equal(np.tril(cov.cpu().numpy()), want)


def _spectrum(ctx, Wt):
    s = min(Wt.shape)
    sig = torch.empty(s, device="cuda")
    vec = torch.empty((s, s), device="cuda")
    sw = torch.zeros(1, dtype=torch.int32, device="cuda")
    K().whitened_svd(ctx, [to_dev(Wt.astype(np.float32), torch)], [sig], [vec], sweeps=sw)
    ctx.sync_status()
    return sig.cpu().numpy(), vec.cpu().numpy(), int(sw.item())


def test_zero_and_rank_one_spectra(ctx):
    sig, vec, sw = _spectrum(ctx, np.zeros((70, 40)))
    assert np.all(sig == 0.0) and sw <= 1
    r = np.random.default_rng(3)
    u, v = r.standard_normal(70), r.standard_normal(40)
    Wt = np.outer(u, v)
    sig, vec, _ = _spectrum(ctx, Wt)
    s0 = np.linalg.norm(u) * np.linalg.norm(v)
    assert abs(sig[0] - s0) <= 1e-5 * s0
    assert np.all(np.abs(sig[1:]) <= 1e-3 * s0)


@pytest.mark.parametrize("m,n", [(1, 40), (40, 1), (1, 1)])
def test_vector_shaped_layers(ctx, m, n):
    r = np.random.default_rng(m * 100 + n)
    A = r.standard_normal((300, m)).astype(np.float32)
    Gr = r.standard_normal((300, n)).astype(np.float32)
    X = O.finalize_covariance(O.covariance_sum(A), 300, 1e-2).astype(np.float32)
    G = O.finalize_covariance(O.covariance_sum(Gr), 300, 1e-2).astype(np.float32)
    W = (r.standard_normal((m, n)) * 0.02).astype(np.float32)
    s = 1
    Sx = torch.empty((m, m), device="cuda")
    Sg = torch.empty((n, n), device="cuda")
    Si = torch.empty((s, s), device="cuda")
    Wt = torch.empty((m, n), device="cuda")
    K().whiten(ctx, to_dev(X, torch), to_dev(G, torch), to_dev(W, torch), Sx, Sg, Si, Wt)
    ctx.sync_status()
    oSx, oSg = O.cholesky_factors(X.astype(np.float64), G.astype(np.float64))
    oWt = O.whiten(W, oSx, oSg)
    assert rel_fro(Wt.cpu().numpy(), oWt) <= 1e-5
    sig = torch.empty(1, device="cuda")
    vec = torch.empty((1, 1), device="cuda")
    K().whitened_svd(ctx, [Wt], [sig], [vec])
    ctx.sync_status()
    assert abs(sig.item() - np.linalg.norm(oWt)) <= 1e-5 * np.linalg.norm(oWt)
    U = torch.empty((m, 1), device="cuda")
    V = torch.empty((1, n), device="cuda")
    K().unwhiten(ctx, to_dev(W, torch), Sx, Sg, Si, sig, vec, 1, U, V)
    ctx.sync_status()
    # full rank: U V reproduces W up to the unwhitening's operand split (hi + lo bfloat16
    # planes, 16 significant bits, about 1.5e-5 relative per operand and product)
    np.testing.assert_allclose(U.cpu().numpy() @ V.cpu().numpy(), W, rtol=0, atol=1e-4 * np.abs(W).max())


def test_allocation_empty_pool_and_extreme_budgets(ctx):
    r = np.random.default_rng(8)
    sig = [np.sort(r.gamma(1.0, 1.0, 30))[::-1].astype(np.float32), np.sort(r.gamma(1.0, 1.0, 12))[::-1].astype(np.float32)]
    costs = [50, 20]
    s = torch.from_numpy(np.concatenate(sig)).cuda()
    off = torch.tensor([0, 30, 42], dtype=torch.int64, device="cuda")
    cost = torch.tensor(costs, dtype=torch.int64, device="cuda")
    for budget in (0, 19, 20, 49, 10 ** 12):
        want = list(O.allocate(sig, costs, budget, precision="f32").ranks)
        if budget == 0:
            assert want == [0, 0]
        if budget == 10 ** 12:
            assert want == [30, 12]
        ranks = torch.full((2,), -1, dtype=torch.int32, device="cuda")
        used = torch.zeros(1, dtype=torch.int64, device="cuda")
        K().score_and_allocate(ctx, s, off, cost, budget, ranks, used=used)
        ctx.sync_status()
        assert ranks.cpu().tolist() == want
        assert int(used.item()) == sum(w * c for w, c in zip(want, costs))
    # an empty pool: every rank 0, no cut
    ranks = torch.full((2,), -1, dtype=torch.int32, device="cuda")
    cut = torch.zeros(2, device="cuda")
    empty = torch.empty(0, device="cuda")
    K().score_and_allocate(ctx, empty, torch.zeros(3, dtype=torch.int64, device="cuda"), cost, 100, ranks, cut=cut)
    ctx.sync_status()
    assert ranks.cpu().tolist() == [0, 0] and np.all(np.isnan(cut.cpu().numpy()))


def test_unwhiten_rank_zero_is_a_no_op(ctx):
    W = torch.zeros((8, 6), device="cuda")
    Sx = torch.eye(8, device="cuda")
    Sg = torch.eye(6, device="cuda")
    Si = torch.eye(6, device="cuda")
    sig = torch.ones(6, device="cuda")
    vec = torch.eye(6, device="cuda")
    U = torch.empty((8, 1), device="cuda")[:, :0]
    V = torch.empty((1, 6), device="cuda")[:0]
    K().unwhiten(ctx, W, Sx, Sg, Si, sig, vec, 0, U, V)
    ctx.sync_status()
