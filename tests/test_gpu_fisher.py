"""LASER Methodology 2's empirical-Fisher component scores on the GPU against the fp64
oracle, the allocation over given keys (bit-identical, with the keep mask), and the whole
pipeline with score="empirical_fisher" on a small block.

Tolerances: the projections a_t . u_i and g_t . v_i run on the tensor cores with U and V split
into hi + lo bfloat16 planes (16 significant bits, about 1.5e-5 relative per operand), so a
score (a product of two squared projections) carries a relative error of order 1e-4; the
tests allow 1e-3, and rank differences only between components whose oracle scores lie
within 1e-3 of the cut.
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


@pytest.mark.parametrize("N,m,n,r,dtype", [(1500, 320, 192, 50, "bf16"), (5000, 257, 130, 130, "bf16"),
                                           (900, 64, 96, 64, "f32")])
def test_empirical_fisher_scores(ctx, N, m, n, r, dtype):
    rng = np.random.default_rng(N + m)
    A = rng.standard_normal((N, m)).astype(np.float32)
    Gr = (rng.standard_normal((N, n)) * 1e-3).astype(np.float32)
    if dtype == "bf16":
        A = recipes.philox.bf16_bits_to_f32(recipes.philox.f32_to_bf16_bits(A))
        Gr = recipes.philox.bf16_bits_to_f32(recipes.philox.f32_to_bf16_bits(Gr))
        Ad, Gd = bf16_dev(A, torch), bf16_dev(Gr, torch)
    else:
        Ad, Gd = to_dev(A, torch), to_dev(Gr, torch)
    U = (rng.standard_normal((m, r)) * 0.05).astype(np.float32)
    V = (rng.standard_normal((r, n)) * 0.05).astype(np.float32)
    acc = torch.zeros(r, dtype=torch.float64, device="cuda")
    K().empirical_fisher_accumulate(ctx, Ad, Gd, to_dev(U, torch), to_dev(V, torch), acc)
    ctx.sync_status()
    got = acc.cpu().numpy() / (2.0 * N)
    want = O.empirical_fisher_scores(A, Gr, U, V)
    assert np.max(np.abs(got / want - 1.0)) <= 1e-3


def test_allocation_over_given_keys(ctx):
    rng = np.random.default_rng(4)
    keys, costs = [], []
    for u in range(30):
        k = int(rng.integers(5, 900))
        keys.append(rng.gamma(0.7, 1.0, k).astype(np.float32))     # not monotone within a unit
        costs.append(int(rng.integers(20, 2000)))
    keys[5][:] = np.round(keys[5], 1)                                # ties
    budget = int(0.3 * sum(len(k) * c for k, c in zip(keys, costs)))
    kd = torch.from_numpy(np.concatenate(keys)).cuda()
    off = torch.tensor([0] + list(np.cumsum([len(k) for k in keys])), dtype=torch.int64, device="cuda")
    cost = torch.tensor(costs, dtype=torch.int64, device="cuda")
    ranks = torch.empty(len(keys), dtype=torch.int32, device="cuda")
    keep = torch.empty(kd.numel(), dtype=torch.uint8, device="cuda")
    cut = torch.empty(2, device="cuda")
    used = torch.zeros(1, dtype=torch.int64, device="cuda")
    K().score_and_allocate_keys(ctx, kd, off, cost, budget, ranks, keep=keep, cut=cut, used=used)
    ctx.sync_status()
    al = O.allocate_keys(keys, costs, budget)
    np.testing.assert_array_equal(ranks.cpu().numpy(), al.ranks)
    assert int(used.item()) == al.used
    want = np.zeros(kd.numel(), dtype=np.uint8)
    offs = np.concatenate([[0], np.cumsum([len(k) for k in keys])])
    n_keep = int(al.ranks.sum())
    want[offs[al.order_unit[:n_keep]] + al.order_comp[:n_keep]] = 1
    np.testing.assert_array_equal(keep.cpu().numpy(), want)


@pytest.mark.parametrize("name", ["mini_block", "mini_vlm_heads_qaw"])
def test_end_to_end_empirical_fisher(ctx, name):
    from synth import device
    from vlm_compression_fac_b300 import pipeline
    wl = recipes.mini_block(n_tokens=1100, seed=95) if name == "mini_block" else recipes.mini_vlm(n_tokens=700)
    quant = wl.quant == "int8_token"
    units = pipeline.unit_specs(wl)
    weights = device.weights_on_device(wl, torch)
    acts = {n: device.stream_on_device(wl, s, 0, wl.n_tokens, torch) for n, s in wl.sites.items() if s.kind == "act"}
    grads = {n: device.stream_on_device(wl, s, 0, wl.n_tokens, torch) for n, s in wl.sites.items() if s.kind == "grad"}
    res = pipeline.compress(ctx, units, weights, acts, grads, wl.n_tokens, lam=wl.lam, budget=wl.budget,
                            quant=quant, score="empirical_fisher")
    ctx.sync_status()
    ref = O.compress_workload(wl)
    keys = [g.scores.cpu().numpy() for g in res.units]
    costs = [u.m + u.n for u in wl.units]
    # the oracle's allocation over the GPU's float32 keys is the GPU's, component for component
    al = O.allocate_keys(keys, costs, wl.budget)
    np.testing.assert_array_equal(np.array([int(g.rank) for g in res.units]), al.ranks)
    assert int(res.used.item()) == al.used <= wl.budget
    n_keep = int(al.ranks.sum())
    for ui, g in enumerate(res.units):
        want = np.sort(al.order_comp[:n_keep][al.order_unit[:n_keep] == ui])
        np.testing.assert_array_equal(np.sort(g.kept.cpu().numpy()), want)
    for g, ur, u in zip(res.units, ref["units"], wl.units):
        kept = g.kept.cpu().numpy()
        U, V = g.U.cpu().numpy(), g.V.cpu().numpy()
        # the keys of the kept components are LASER's scores of the GPU's own factors
        A = recipes.gen_stream(wl, wl.sites[u.x_site], 0, wl.n_tokens)
        if quant:
            A = O.fake_quant_int8_token(A)        # over the full width, as for the covariance
        A = A[:, u.x_off:u.x_off + u.m]
        Gr = recipes.gen_stream(wl, wl.sites[u.g_site], 0, wl.n_tokens)[:, u.g_off:u.g_off + u.n]
        if len(kept):
            ko = O.empirical_fisher_scores(A, Gr, U, V)
            kg = g.scores.cpu().numpy().astype(np.float64)[kept]
            assert np.max(np.abs(kg - ko) / np.maximum(ko, 1e-6 * ko.max())) <= 1e-3, g.name
        # the whitened error of any kept subset is the sum of the dropped sigma^2
        dropped = np.setdiff1d(np.arange(len(ur.sigma)), kept)
        e = O.whitened_error(recipes.gen_weight(wl, u), U, V, ur.Sx, ur.Sg)
        e_want = float(np.sum(g.sigma.cpu().numpy().astype(np.float64)[dropped] ** 2))
        tot = float(np.sum(ur.sigma ** 2))
        assert abs(e - e_want) <= 1e-3 * max(e_want, 1e-6 * tot), (g.name, e, e_want)


def test_end_to_end_energy_ratio_with_layer_weights(ctx):
    from synth import device
    from vlm_compression_fac_b300 import pipeline
    wl = recipes.mini_block(n_tokens=1100, seed=96)
    units = pipeline.unit_specs(wl)
    weights = device.weights_on_device(wl, torch)
    acts = {n: device.stream_on_device(wl, s, 0, wl.n_tokens, torch) for n, s in wl.sites.items() if s.kind == "act"}
    grads = {n: device.stream_on_device(wl, s, 0, wl.n_tokens, torch) for n, s in wl.sites.items() if s.kind == "grad"}
    uw = [0.5 + 0.25 * i for i in range(len(units))]
    res = pipeline.compress(ctx, units, weights, acts, grads, wl.n_tokens, lam=wl.lam, budget=wl.budget,
                            score="energy_ratio", unit_weights=uw)
    ctx.sync_status()
    sig = [g.sigma.cpu().numpy() for g in res.units]
    costs = [u.m + u.n for u in wl.units]
    al = O.allocate(sig, costs, wl.budget, mode=O.KEY_ENERGY_RATIO, precision="f32", weights=uw)
    np.testing.assert_array_equal(np.array([int(g.rank) for g in res.units]), al.ranks)
    assert int(res.used.item()) == al.used <= wl.budget
    for g in res.units:
        assert g.U.shape[1] == g.rank and g.V.shape[0] == g.rank


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_fake_quant_rows_bit_exact(ctx, dtype):
    rng = np.random.default_rng(12)
    A = (rng.standard_normal((257, 136)) * rng.gamma(1.0, 1.0, (257, 1))).astype(np.float32)
    A[3] = 0.0
    A[7, 5] = -40.0
    if dtype == "bf16":
        A = recipes.philox.bf16_bits_to_f32(recipes.philox.f32_to_bf16_bits(A))
        Ad = bf16_dev(A, torch)
    else:
        Ad = to_dev(A, torch)
    out = torch.empty(A.shape, dtype=torch.bfloat16, device="cuda")
    K().fake_quant_rows(ctx, Ad, out)
    ctx.sync_status()
    np.testing.assert_array_equal(out.float().cpu().numpy(), O.fake_quant_int8_token(A))
