"""GPU tests of Swift-SVD's hybrid allocation key and of a device-side wait that runs out.

* score_and_allocate_hybrid (Swift-SVD section B, hybrid scoring beta^alpha log(e + eps*)^(1-alpha)
  per component) against the oracle's keys and sort-and-truncate on the same float32 spectra:
  identical ranks and used parameters, cut scores within one float32 ulp (the keys go through
  float64 log and pow, whose last bit may differ between libraries; the float32 rounding
  absorbs that except within 2^-29 of a rounding boundary);
* the pipeline with score="swift_hybrid" end to end on a small block against the oracle;
* kf_set_wait_limit: a tensor-core SYRK whose pipeline waits are limited to 100 ns gives up,
  reports KF_ERR_TIMEOUT through kf_sync_status without faulting, and the next call on the
  same context with the default limit is correct (the bounded-wait failure path).
"""
import numpy as np
import pytest

import oracle as O
from synth import recipes
from tests.gpu_util import bf16_dev, lower, rank_parity, rel_fro

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


def _ulp_close(a, b):
    if np.isnan(a) or np.isnan(b):
        return np.isnan(a) and np.isnan(b)
    fa, fb = np.float32(a), np.float32(b)
    return fa == fb or np.nextafter(fa, np.float32(np.inf)) == fb or np.nextafter(fa, np.float32(-np.inf)) == fb


HYBRID_CASES = [  # (n_units, max_len, budget fraction, alpha, ties)
    (40, 600, 0.35, 0.5, False),
    (40, 600, 0.35, 0.0, False),
    (40, 600, 0.2, 1.0, False),
    (12, 64, 0.4, 0.3, True),
    (60, 4100, 0.4, 0.75, False),   # ~120k components: many radix tiles
]


@pytest.mark.parametrize("case", HYBRID_CASES)
def test_swift_hybrid_allocation_matches_the_oracle(ctx, case):
    nu, ml, frac, alpha, ties = case
    r = np.random.default_rng(nu * 7 + ml)
    sig, costs = [], []
    for u in range(nu):
        m, n = int(r.integers(8, ml + 8)), int(r.integers(8, ml + 8))
        s = np.sort(r.gamma(1.0, 1.0, size=min(m, n)))[::-1].astype(np.float32)
        if ties:   # identical spectra in pairs of units: equal keys across units (lower unit first)
            s = np.round(s, 1).astype(np.float32)
            if u % 2 == 1:
                s = sig[-1].copy()
                m, n = costs[-1] // 2, costs[-1] - costs[-1] // 2
        sig.append(s)
        costs.append(m + n)
    beta = r.uniform(0.1, 2.0, nu).astype(np.float32)
    beta[2] = 0.0
    if ties:
        beta[:] = 1.0
    budget = int(frac * sum(len(s) * c for s, c in zip(sig, costs)))
    sd = torch.from_numpy(np.concatenate(sig)).cuda()
    off = torch.tensor([0] + list(np.cumsum([len(s) for s in sig])), dtype=torch.int64, device="cuda")
    cost = torch.tensor(costs, dtype=torch.int64, device="cuda")
    ranks = torch.empty(nu, dtype=torch.int32, device="cuda")
    cut = torch.empty(2, dtype=torch.float32, device="cuda")
    used = torch.zeros(1, dtype=torch.int64, device="cuda")
    K().score_and_allocate_hybrid(ctx, sd, off, cost, budget, ranks, alpha, importance=torch.from_numpy(beta).cuda(),
                                  cut=cut, used=used)
    ctx.sync_status()
    al = O.allocate_swift_hybrid(sig, costs, budget, list(beta), alpha)
    np.testing.assert_array_equal(ranks.cpu().numpy(), al.ranks)
    assert int(used.item()) == al.used <= budget
    c = cut.cpu().numpy()
    assert _ulp_close(c[0], al.cut_score) and _ulp_close(c[1], al.next_score), (c, al.cut_score, al.next_score)


def test_swift_hybrid_alpha_is_checked(ctx):
    z = torch.zeros(4, dtype=torch.float32, device="cuda")
    off = torch.tensor([0, 4], dtype=torch.int64, device="cuda")
    cost = torch.tensor([3], dtype=torch.int64, device="cuda")
    ranks = torch.empty(1, dtype=torch.int32, device="cuda")
    with pytest.raises(K().KfsvdError):
        K().score_and_allocate_hybrid(ctx, z, off, cost, 5, ranks, -0.1)


def test_end_to_end_swift_hybrid(ctx):
    """compress(score="swift_hybrid") on a small block: the oracle's hybrid allocation fed the
    GPU's float32 spectra gives the GPU's ranks, and against the oracle's own spectra the
    ranks differ at most at keys within 1e-6 of the cut; the factors match the optimum."""
    from synth import device
    from vlm_compression_fac_b300 import pipeline
    wl = recipes.mini_block()
    beta = [1.0, 0.5, 2.0, 1.0, 1.5, 0.8, 1.2][:len(wl.units)]
    alpha = 0.6
    units = pipeline.unit_specs(wl)
    weights = device.weights_on_device(wl, torch)
    acts = {n: device.stream_on_device(wl, s, 0, wl.n_tokens, torch) for n, s in wl.sites.items() if s.kind == "act"}
    grads = {n: device.stream_on_device(wl, s, 0, wl.n_tokens, torch) for n, s in wl.sites.items()
             if s.kind == "grad"}
    res = pipeline.compress(ctx, units, weights, acts, grads, wl.n_tokens, lam=wl.lam, budget=wl.budget,
                            score="swift_hybrid", unit_weights=beta, alpha=alpha)
    ctx.sync_status()
    ref = O.compress_workload(wl)
    costs = [u.m + u.n for u in wl.units]
    sig_g = [u.sigma.cpu().numpy() for u in res.units]
    al32 = O.allocate_swift_hybrid(sig_g, costs, wl.budget, beta, alpha)
    ranks = res.ranks.cpu().numpy()
    np.testing.assert_array_equal(ranks, al32.ranks)
    alo = O.allocate_swift_hybrid([o.sigma.astype(np.float32) for o in ref["units"]], costs, wl.budget, beta, alpha)
    keys_o = [O.swift_hybrid_keys(o.sigma.astype(np.float32), b, alpha).astype(np.float64)
              for o, b in zip(ref["units"], beta)]
    cut = alo.cut_score if np.isfinite(alo.cut_score) else alo.next_score
    for u, (rg, ro) in enumerate(zip(ranks, alo.ranks)):
        for i in range(min(rg, ro), max(rg, ro)):
            assert abs(keys_o[u][i] - cut) <= 1e-6 * abs(cut), (u, i)
    for g, o in zip(res.units, ref["units"]):
        W = recipes.gen_weight(wl, [x for x in wl.units if x.name == g.name][0])
        e = O.whitened_error(W, g.U.cpu().numpy(), g.V.cpu().numpy(), o.Sx, o.Sg)
        e_opt = float(np.sum(o.sigma[g.rank:] ** 2))
        assert e_opt <= 1e-12 * float(np.sum(o.sigma ** 2)) or abs(e / e_opt - 1.0) <= 1e-3, g.name


def test_short_wait_limit_times_out_and_the_context_recovers(ctx):
    """A device-side wait that runs out: with every tensor-core pipeline wait limited to 100 ns,
    a covariance SYRK over 65536 tokens gives up (KF_ERR_TIMEOUT with a wait-site code, read by
    kf_sync_status); no fault, no hang (the kernel drains what it issued on the long limit).
    With the default limit restored, the same context computes the covariance correctly."""
    d, n_tok = 256, 65536
    wl = recipes.mini_block(n_tokens=n_tok, d=d, ffn=704)
    A = recipes.gen_stream(wl, wl.sites["attn_in"], 0, n_tok)
    Ad = bf16_dev(A, torch)
    seen = None
    try:
        K().kf_set_wait_limit(ctx, 100)
        for _ in range(3):
            cov = torch.zeros((d, d), dtype=torch.float32, device="cuda")
            K().kfac_accumulate(ctx, Ad, cov)
            try:
                ctx.sync_status()
            except K().KfsvdError as e:
                seen = e
                break
    finally:
        K().kf_set_wait_limit(ctx, 0)
    assert seen is not None and seen.status == K().KF_ERR_TIMEOUT, seen
    assert "timed out" in str(seen)
    cov = torch.zeros((d, d), dtype=torch.float32, device="cuda")
    K().kfac_accumulate(ctx, Ad, cov)
    ctx.sync_status()
    assert rel_fro(lower(cov.cpu().numpy()), lower(O.covariance_sum(A))) <= 1e-4
