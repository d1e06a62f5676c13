"""Full-size runs of the other synthetic workloads, through the streaming pipeline, with
per-unit parity against the oracle:

  * 70B-shaped block (d 8192, FFN 28672, GQA k/v 8192x1024, N = 262144, 30% kept): every unit;
  * 32-block 7B-shaped model (224 matrices, N = 65536 per layer, per-layer seeds, 40% kept
    globally; processed block by block): every unit of the first block;
  * VLM-shaped (ViT-L 24 blocks + 28-block LM with 128-dim heads as units, GQA, N = 147456,
    INT8 per-token fake-quantised activations, one 50% pool of 677,888 components): every unit
    of the first ViT block (6 matrices), all 64 attention heads of the first LM block and that
    block's FFN (gate, up, down).

Per checked unit (step parity: the oracle, in float64, takes the GPU's finalised factors X and
G as its inputs, computes S_x, S_g, W~ = S_x W S_g and the spectrum by eigh of the Gram):
|sigma - sigma_oracle| <= 1e-3 sigma_max, and the whitened error of the GPU's U V against the
optimum at the same rank within 1e-3.  Covariances: sampled entries against float64 sums over
all N tokens of the generator's columns (relative 1e-4 of the entry's scale).

Ranks: the oracle's allocation fed the GPU's float32 spectra is bit-identical (the sort and
the cut).  For the 70B block every unit's oracle spectrum is known and the ranks must equal the
oracle's except at score ties within 1e-6 of the cut.  For the 32-block model and the VLM
(~10^6 components in one pool) the oracle's spectra cannot all be computed inside a test, and
the float32 W~ (about 1e-6 relative) already limits sigma near the cut to about the measured
error delta (the largest relative sigma error of the checked units over their kept components
and the next 16).  The check there is a margin argument: the oracle spectra of the checked units
and of the band units closest to the cut replace the GPU's, and every component on which the
resulting allocation and the GPU's differ must have its score within the band (1 + 2 delta)^2
of the cut, i.e. every rank difference is explained by the measured sigma error.  The band
size, the recomputed units and the moved components are printed.
"""
import time

import numpy as np
import pytest

import oracle as O
from synth import recipes
from tests.gpu_util import host_weight, rank_parity

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

MAX_RECHECK_UNITS = 8


def _entry_sum(wl, site, i, j, chunk=65536):
    s = 0.0
    for t0 in range(0, wl.n_tokens, chunk):
        A = recipes.gen_stream(wl, site, t0, min(wl.n_tokens, t0 + chunk), cols=[i, j]).astype(np.float64)
        if wl.quant == "int8_token" and site.kind == "act":
            raise ValueError("entry sums of quantised streams need whole rows")
        s += float(A[:, 0] @ A[:, 1])
    return s


def _run(wl, keep_sites, keep_units, groups_by_block):
    from synth import device
    from vlm_compression_fac_b300 import kfsvd as K, pipeline
    ctx = K.Context(0)
    units = pipeline.unit_specs(wl)
    weights = device.weights_on_device(wl, torch)
    groups = None
    if groups_by_block:
        blocks = sorted({u.block for u in wl.units})
        groups = [[i for i, u in enumerate(wl.units) if u.block == b] for b in blocks]
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    res = pipeline.compress(ctx, units, weights, device.rows_fn(wl, torch), None, wl.n_tokens, lam=wl.lam,
                            budget=wl.budget, quant=wl.quant == "int8_token",
                            site_dims={n: s.d for n, s in wl.sites.items()},
                            act_sites=[n for n, s in wl.sites.items() if s.kind == "act"],
                            groups=groups, chunk_tokens=32768, keep_covs=list(keep_sites), keep_whitened=False)
    ctx.sync_status()
    secs = time.perf_counter() - t0
    out = {
        "secs": secs,
        "covs": {k: v.cpu().numpy() for k, v in res.covs.items()},
        "sigma": [u.sigma.cpu().numpy() for u in res.units],
        "ranks": res.ranks.cpu().numpy(),
        "used": int(res.used.item()),
        "cut": res.cut.cpu().numpy(),
        "sweeps": [u.sweeps for u in res.units],
    }
    names = [u.name for u in wl.units]
    out["factors"] = {n: (res.units[names.index(n)].U.cpu().numpy(), res.units[names.index(n)].V.cpu().numpy())
                      for n in keep_units}
    del res, weights
    ctx.close()
    torch.cuda.empty_cache()
    print("%s: %d units, %.1f s end to end on the GPU, sweeps %d..%d" % (
        wl.name, len(wl.units), secs, min(out["sweeps"]), max(out["sweeps"])))
    return out


def _check_allocation(wl, out):
    costs = [u.m + u.n for u in wl.units]
    al32 = O.allocate(out["sigma"], costs, wl.budget, precision="f32")
    np.testing.assert_array_equal(out["ranks"], al32.ranks)
    assert out["used"] == al32.used
    assert out["used"] <= wl.budget
    for r, s in zip(out["ranks"], out["sigma"]):
        assert 0 <= r <= len(s)
        assert np.all(np.diff(s) <= 0)


def _site_cov(wl, out, name):
    """A site's finalised float32 factor as the pipeline built it: kept from the run, or built
    again by the same library calls (kfac_accumulate over the same generated rows in the same
    chunks, then kf_finalize_covariance; deterministic, so identical to the run's)."""
    if name in out["covs"]:
        return out["covs"][name]
    from synth import device
    from vlm_compression_fac_b300 import kfsvd as K
    site = wl.sites[name]
    ctx = K.Context(0)
    cov = torch.zeros((site.d, site.d), dtype=torch.float32, device="cuda")
    q = K.KF_QUANT_INT8_TOKEN if (wl.quant == "int8_token" and site.kind == "act") else K.KF_QUANT_NONE
    for t0 in range(0, wl.n_tokens, 32768):
        rows = device.stream_on_device(wl, site, t0, min(wl.n_tokens, t0 + 32768), torch)
        K.kfac_accumulate(ctx, rows, cov, quant=q)
        del rows
    K.kf_finalize_covariance(ctx, cov, wl.n_tokens, wl.lam)
    ctx.sync_status()
    out["covs"][name] = cov.cpu().numpy()
    del cov
    ctx.close()
    torch.cuda.empty_cache()
    return out["covs"][name]


def _oracle_sigma(wl, out, i):
    """The oracle's spectrum of unit i from the GPU's finalised factors (step parity), and the
    oracle factors needed for the whitened error."""
    u = wl.units[i]
    X = _site_cov(wl, out, u.x_site).astype(np.float64)[u.x_off:u.x_off + u.m, u.x_off:u.x_off + u.m]
    G = _site_cov(wl, out, u.g_site).astype(np.float64)[u.g_off:u.g_off + u.n, u.g_off:u.g_off + u.n]
    Sx, Sg = O.cholesky_factors(X, G)
    del X, G
    W = host_weight(wl, u, torch, out.setdefault("wcache", {})).astype(np.float64)
    Wt = O.whiten(W, Sx, Sg)
    so = np.sqrt(np.maximum(O.gram_eigenvalues(Wt), 0.0))
    return so, (W, Sx, Sg, Wt)


def _check_units(wl, out, names, oracle_sig):
    """sigma within 1e-3 sigma_max and the whitened-error ratio within 1e-3 on every named
    unit; records each unit's oracle spectrum.  Returns the largest relative sigma error over
    the kept components and the next 16."""
    idx = {u.name: i for i, u in enumerate(wl.units)}
    worst = 0.0
    problems = []
    t0 = time.perf_counter()
    for name in names:
        i = idx[name]
        so, (W, Sx, Sg, Wt) = _oracle_sigma(wl, out, i)
        oracle_sig[i] = so
        sg = out["sigma"][i].astype(np.float64)
        if np.max(np.abs(sg - so)) > 1e-3 * so[0]:
            problems.append(("sigma", name, float(np.max(np.abs(sg - so)) / so[0])))
        r = int(out["ranks"][i])
        k = min(len(so), r + 16)
        nz = so[:k] > 0
        if np.any(nz):
            worst = max(worst, float(np.max(np.abs(sg[:k][nz] / so[:k][nz] - 1.0))))
        if name in out["factors"]:
            U, V = out["factors"][name]
            e_opt = float(np.sum(so[r:] ** 2))
            # ||S_x (W - U V) S_g||^2 = ||W~ - (S_x U)(V S_g)||^2
            D = Wt - (Sx @ U.astype(np.float64)) @ (V.astype(np.float64) @ Sg)
            e = float(np.sum(D * D))
            if e_opt > 1e-12 * float(np.sum(so ** 2)) and abs(e / e_opt - 1.0) > 1e-3:
                problems.append(("whitened error", name, e, e_opt))
        del W, Sx, Sg, Wt
    print("%s: %d units checked against the oracle in %.1f s" % (wl.name, len(names), time.perf_counter() - t0))
    assert not problems, problems
    return worst


def _check_ranks_by_margin(wl, out, oracle_sig, delta):
    """Rank parity against the oracle's own spectra by the margin argument in the module
    docstring: the oracle spectra of the checked units and of up to MAX_RECHECK_UNITS more band
    units (closest to the cut first) replace the GPU's; the rest of the band is reported.
    Returns (band size, recomputed units)."""
    costs = [u.m + u.n for u in wl.units]
    al = O.allocate(out["sigma"], costs, wl.budget, precision="f32")
    c_last = al.cut_score if np.isfinite(al.cut_score) else al.next_score
    c_next = al.next_score if np.isfinite(al.next_score) else al.cut_score
    f = (1.0 + 2.0 * max(delta, 1e-7)) ** 2
    lo, hi = c_next / f, c_last * f
    band_units = {}
    band = 0
    cut = 0.5 * (c_last + c_next)
    for i, s in enumerate(out["sigma"]):
        sc = 0.5 * s.astype(np.float64) ** 2
        m = (sc * f >= lo) & (sc / f <= hi)
        if np.any(m):
            band += int(np.sum(m))
            band_units[i] = float(np.min(np.abs(sc[m] / cut - 1.0)))
    # recompute the units whose band components lie closest to the cut first
    todo = sorted((i for i in band_units if i not in oracle_sig), key=lambda i: band_units[i])
    done = todo[:MAX_RECHECK_UNITS]
    t0 = time.perf_counter()
    for i in done:
        oracle_sig[i], _ = _oracle_sigma(wl, out, i)
    print("%s: %d band units recomputed by the oracle in %.1f s" % (wl.name, len(done), time.perf_counter() - t0))
    left = len(todo) - len(done)
    print("%s: delta %.2e, %d components of %d units in the cut band; oracle spectra for %d of them (%d checked "
          "units, %d recomputed closest to the cut); %d band units keep their GPU spectra (ranks there rest on the "
          "measured error bound)" % (wl.name, delta, band, len(band_units),
                                     len([i for i in band_units if i in oracle_sig]), len(oracle_sig) - len(done),
                                     len(done), left))
    mixed = [oracle_sig[i] if i in oracle_sig else out["sigma"][i].astype(np.float64)
             for i in range(len(wl.units))]
    ref = O.allocate(mixed, costs, wl.budget)
    ok, moved = rank_parity(out["ranks"], ref, mixed, (1.0 + 2.0 * max(delta, 1e-7)) ** 2 - 1.0)
    smax = max(0.5 * float(np.max(x)) ** 2 for x in mixed)
    print("%s: %d components move against the allocation with oracle spectra substituted; farthest from "
          "the cut %.2e relative to the cut score, %.2e relative to the largest score" % (
              wl.name, len(moved), max([d for _, _, d in moved], default=0.0),
              max([d for _, _, d in moved], default=0.0) * abs(cut) / smax))
    assert ok, moved
    return band, done


def _check_cov_entries(wl, out, site_name, pairs):
    site = wl.sites[site_name]
    C = out["covs"][site_name].astype(np.float64)
    N = wl.n_tokens
    for i, j in pairs:
        S_ij = _entry_sum(wl, site, i, j)
        S_ii = _entry_sum(wl, site, i, i)
        S_jj = _entry_sum(wl, site, j, j)
        assert abs(C[i, j] - S_ij / N) <= 1e-4 * np.sqrt(S_ii * S_jj) / N, (site_name, i, j)


def test_llama70b_block_every_unit():
    wl = recipes.llama70b_block()
    names = [u.name for u in wl.units]
    out = _run(wl, list(wl.sites), names, False)
    _check_allocation(wl, out)
    _check_cov_entries(wl, out, "attn_in", [(0, 1), (8191, 77), (int(recipes.outlier_channels(wl, wl.sites["attn_in"])[0]), 5)])
    _check_cov_entries(wl, out, "gate_out", [(0, 28671), (12345, 54)])
    oracle_sig = {}
    delta = _check_units(wl, out, names, oracle_sig)
    # every unit has its oracle spectrum: the ranks are compared directly
    costs = [u.m + u.n for u in wl.units]
    ref = O.allocate([oracle_sig[i] for i in range(len(names))], costs, wl.budget)
    ok, moved = rank_parity(out["ranks"], ref, [oracle_sig[i] for i in range(len(names))], 1e-6)
    print("llama70b_block: max relative sigma error over kept components %.2e; ranks %s" % (delta, list(out["ranks"])))
    assert ok, moved


def test_llama7b_model_32_blocks_whole_block():
    wl = recipes.llama7b_model()
    assert len(wl.units) == 224
    first = [u.name for u in wl.units if u.block == 0]
    sites = sorted({s for u in wl.units if u.block == 0 for s in (u.x_site, u.g_site)})
    out = _run(wl, sites, first, True)
    _check_allocation(wl, out)
    _check_cov_entries(wl, out, "b0.attn_in", [(0, 1), (4095, 17)])
    oracle_sig = {}
    delta = _check_units(wl, out, first, oracle_sig)
    _check_ranks_by_margin(wl, out, oracle_sig, delta)


def test_vlm_heads_qaw_first_blocks():
    wl = recipes.vlm()
    assert sum(min(u.m, u.n) for u in wl.units) == 677888
    vit0 = [u.name for u in wl.units if u.name.startswith("vit.b0.")]
    lm0 = [u.name for u in wl.units if u.name.startswith("lm.b0.")]
    assert len(vit0) == 6 and len(lm0) == 64 + 3
    sites = sorted({s for u in wl.units if u.name in set(vit0 + lm0) for s in (u.x_site, u.g_site)})
    out = _run(wl, sites, vit0 + lm0, True)
    _check_allocation(wl, out)
    oracle_sig = {}
    delta = _check_units(wl, out, vit0 + lm0, oracle_sig)
    _check_ranks_by_margin(wl, out, oracle_sig, delta)
    # quantisation-aware covariance at full width on a 4096-token slice of the same stream
    from synth import device
    from vlm_compression_fac_b300 import kfsvd as K
    site = wl.sites["vit.b0.attn_in"]
    A = recipes.gen_stream(wl, site, 0, 4096)
    ctx = K.Context(0)
    cov = torch.zeros((site.d, site.d), dtype=torch.float32, device="cuda")
    K.kfac_accumulate(ctx, device.stream_on_device(wl, site, 0, 4096, torch), cov, quant=K.KF_QUANT_INT8_TOKEN)
    ctx.sync_status()
    want = O.covariance_sum(O.fake_quant_int8_token(A))
    got = np.tril(cov.cpu().numpy().astype(np.float64))
    assert np.linalg.norm(got - np.tril(want)) <= 1e-4 * np.linalg.norm(np.tril(want))
    ctx.close()
