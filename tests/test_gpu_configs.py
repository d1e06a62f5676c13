"""Full-size runs of the other synthetic workloads, through the streaming pipeline, with the
checks the oracle can afford at that size:

  * 70B-shaped block (d 8192, FFN 28672, GQA k/v 8192x1024, N = 262144, 30% kept);
  * 32-block 7B-shaped model (224 matrices, N = 65536 per layer, per-layer seeds, 40% kept
    globally; processed block by block);
  * VLM-shaped (ViT-L 24 blocks + 28-block LM with 128-dim heads as units, GQA, N = 147456,
    INT8 per-token fake-quantised activations, one 50% pool of 677,888 components).

Per workload: sampled covariance entries against float64 sums over all N tokens; step parity
of representative units (the oracle, in float64, takes the GPU's finalised factors as its
inputs: factors, W~, spectrum by eigh of the Gram, whitened error of the GPU's U V); the
oracle's allocation fed the GPU's float32 spectra is bit-identical; the budget holds.
Tolerances as in test_gpu_parity.py.
"""
import time

import numpy as np
import pytest

import oracle as O
from synth import recipes

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def _entry_sum(wl, site, i, j, chunk=65536):
    s = 0.0
    for t0 in range(0, wl.n_tokens, chunk):
        A = recipes.gen_stream(wl, site, t0, min(wl.n_tokens, t0 + chunk), cols=[i, j]).astype(np.float64)
        s += float(A[:, 0] @ A[:, 1])
    return s


def _run(wl, keep_sites, groups_by_block):
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
        "sweeps": [u.sweeps for u in res.units],
    }
    keep = {}
    for i, u in enumerate(wl.units):
        if u.x_site in keep_sites and u.g_site in keep_sites:
            keep[u.name] = (res.units[i].U.cpu().numpy(), res.units[i].V.cpu().numpy())
    out["factors"] = keep
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


def _check_unit(wl, out, name):
    i = [u.name for u in wl.units].index(name)
    u = wl.units[i]
    X = out["covs"][u.x_site].astype(np.float64)[u.x_off:u.x_off + u.m, u.x_off:u.x_off + u.m]
    G = out["covs"][u.g_site].astype(np.float64)[u.g_off:u.g_off + u.n, u.g_off:u.g_off + u.n]
    Sx, Sg = O.cholesky_factors(X, G)
    W = recipes.gen_weight(wl, u).astype(np.float64)
    Wt = O.whiten(W, Sx, Sg)
    so = np.sqrt(np.maximum(O.gram_eigenvalues(Wt), 0.0))
    sg = out["sigma"][i]
    assert np.max(np.abs(sg - so)) <= 1e-3 * so[0], name
    r = int(out["ranks"][i])
    U, V = out["factors"][name]
    e = O.whitened_error(W, U, V, Sx, Sg)
    e_opt = float(np.sum(so[r:] ** 2))
    assert abs(e / e_opt - 1.0) <= 1e-3, (name, e, e_opt)


def _check_cov_entries(wl, out, site_name, pairs):
    site = wl.sites[site_name]
    C = out["covs"][site_name].astype(np.float64)
    N = wl.n_tokens
    for i, j in pairs:
        S_ij = _entry_sum(wl, site, i, j)
        S_ii = _entry_sum(wl, site, i, i)
        S_jj = _entry_sum(wl, site, j, j)
        assert abs(C[i, j] - S_ij / N) <= 1e-4 * np.sqrt(S_ii * S_jj) / N, (site_name, i, j)


def test_llama70b_block():
    wl = recipes.llama70b_block()
    out = _run(wl, ["attn_in", "k_out", "gate_out"], False)
    _check_allocation(wl, out)
    _check_cov_entries(wl, out, "attn_in", [(0, 1), (8191, 77), (int(recipes.outlier_channels(wl, wl.sites["attn_in"])[0]), 5)])
    _check_cov_entries(wl, out, "gate_out", [(0, 28671), (12345, 54)])
    _check_unit(wl, out, "k")


def test_llama7b_model_32_blocks():
    wl = recipes.llama7b_model()
    assert len(wl.units) == 224
    out = _run(wl, ["b0.attn_in", "b0.q_out", "b31.down_in", "b31.down_out"], True)
    _check_allocation(wl, out)
    _check_cov_entries(wl, out, "b0.attn_in", [(0, 1), (4095, 17)])
    _check_unit(wl, out, "b0.q")
    _check_unit(wl, out, "b31.down")


def test_vlm_heads_qaw():
    wl = recipes.vlm()
    assert sum(min(u.m, u.n) for u in wl.units) == 677888
    out = _run(wl, ["lm.b0.attn_in", "lm.b0.q_out", "lm.b0.o_in", "lm.b0.o_out", "vit.b0.attn_in", "vit.b0.q_out"],
               True)
    _check_allocation(wl, out)
    _check_unit(wl, out, "lm.b0.q.h3")
    _check_unit(wl, out, "lm.b0.o.h5")
    _check_unit(wl, out, "vit.b0.q")
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
