"""Whole-workload driver over the C ABI: the call a user makes to compress a set of layers.

For every calibration site it streams the rows into a K-FAC factor (kfac_accumulate) and
finalises it (kf_finalize_covariance); for every unit it whitens W (whiten, sharing a factor
between the units that read the same site); it takes the spectra of the units in batches of
equal min(m, n) (whitened_svd); it allocates ranks globally (score_and_allocate) and maps the
kept factors back (unwhiten).  The only host round trip is reading the per-unit ranks after
the allocation, to size U and V.

A unit may be a block of a larger weight (an attention head): it then reads the rows/columns
of its weight and the diagonal blocks of its factors given by its spec (LASER allocates
across heads; q/k/v heads are column blocks with the head's block of G, o heads row blocks
with the head's block of X).

Calibration rows are either resident device tensors (one per site) or produced on demand by
a callable ``rows(site, t0, t1)``; with ``groups`` the units are processed group by group
(e.g. one transformer block at a time): a group's covariances are built, its units whitened
and their spectra taken, then the covariances and every factor that the unwhitening does not
need are released, so that workloads far larger than device memory stream through.
"""
from __future__ import annotations

import contextlib
from dataclasses import dataclass, field
from typing import Callable, Dict, List, Optional, Sequence, Union

import torch

from . import kfsvd as K


@dataclass
class UnitSpec:
    name: str
    m: int
    n: int
    x_site: str
    g_site: str
    w_name: str = ""      # weight this unit is a block of (empty: the weight `name` itself)
    row0: int = 0
    col0: int = 0
    x_off: int = 0        # diagonal block [x_off, x_off + m) of the input factor
    g_off: int = 0        # diagonal block [g_off, g_off + n) of the output factor

    @property
    def weight(self) -> str:
        return self.w_name or self.name


@dataclass
class UnitOut:
    name: str
    m: int
    n: int
    side: int
    Sx: Optional[torch.Tensor]
    Sg: Optional[torch.Tensor]
    Sinv: torch.Tensor
    Wt: Optional[torch.Tensor]
    sigma: Optional[torch.Tensor] = None
    vecs: Optional[torch.Tensor] = None
    sweeps: int = 0
    rank: int = 0
    U: Optional[torch.Tensor] = None
    V: Optional[torch.Tensor] = None
    kept: Optional[torch.Tensor] = None     # empirical-Fisher allocation: kept component indices
    scores: Optional[torch.Tensor] = None   # empirical-Fisher allocation: the component scores


@dataclass
class Result:
    units: List[UnitOut]
    covs: Dict[str, torch.Tensor]
    ranks: torch.Tensor
    cut: torch.Tensor
    used: torch.Tensor
    timings: Dict[str, float] = field(default_factory=dict)

    def larger_than_dense(self) -> List[str]:
        """Units whose kept factors hold more parameters than the dense weight, r (m + n) > m n.
        The allocation allows this (there is no dense fallback in the path); it is reported."""
        return [u.name for u in self.units if int(u.rank) * (u.m + u.n) > u.m * u.n]


RowsFn = Callable[[str, int, int], torch.Tensor]


def unit_specs(wl) -> List[UnitSpec]:
    """The pipeline's unit specs of a synthetic workload (synth.recipes.Workload)."""
    return [UnitSpec(u.name, u.m, u.n, u.x_site, u.g_site, u.w_name, u.row0, u.col0, u.x_off, u.g_off)
            for u in wl.units]


SCORES = (None, "half_sigma2", "energy_ratio", "empirical_fisher", "swift_hybrid")


def _on_stream(stream):
    """Every library call of a driver runs on ``stream`` and so must the torch operations
    between them (zero fills, slicing, concatenation, the caching allocator's reuse): the
    drivers run under ``torch.cuda.stream(stream)``.  ``stream`` is a torch.cuda.Stream (or
    an ExternalStream wrapping a foreign handle) or None for the current stream."""
    if stream is None:
        return contextlib.nullcontext()
    if not isinstance(stream, torch.cuda.Stream):
        raise TypeError("stream must be a torch.cuda.Stream (torch.cuda.ExternalStream for a raw handle) or None")
    return torch.cuda.stream(stream)


def _allocate(ctx, sig, off, cost, budget, ranks, cut, used, stream, score=None, mode=K.KF_KEY_HALF_SIGMA2,
              fixed_rank=None, unit_weights=None, alpha=None):
    """The global allocation call for the scores that need no second pass over the rows:
    1/2 sigma^2 (``mode`` may pick the per-parameter key), a fixed rank, UniRank's energy ratio
    times ``unit_weights`` (I_l), or Swift-SVD's hybrid score with ``unit_weights`` as the
    layer importance beta and ``alpha``."""
    dev = ranks.device
    w = None if unit_weights is None else torch.tensor([float(x) for x in unit_weights], dtype=torch.float32,
                                                        device=dev)
    if w is not None and w.numel() != ranks.numel():
        raise ValueError("unit_weights: one weight per unit expected")
    if score == "energy_ratio":
        K.score_and_allocate_weighted(ctx, sig, off, cost, int(budget), ranks, mode=K.KF_KEY_ENERGY_RATIO,
                                      unit_weight=w, cut=cut, used=used, stream=stream)
    elif score == "swift_hybrid":
        if alpha is None:
            raise ValueError("score 'swift_hybrid' needs alpha")
        K.score_and_allocate_hybrid(ctx, sig, off, cost, int(budget), ranks, float(alpha), importance=w, cut=cut,
                                    used=used, stream=stream)
    elif fixed_rank is not None:
        fr = torch.full((ranks.numel(),), int(fixed_rank), dtype=torch.int32, device=dev)
        K.score_and_allocate(ctx, sig, off, cost, 0, ranks, mode=K.KF_FIXED_RANK, fixed_rank=fr, cut=cut,
                             used=used, stream=stream)
    else:
        K.score_and_allocate(ctx, sig, off, cost, int(budget), ranks, mode=mode, cut=cut, used=used, stream=stream)


def compress(ctx: K.Context, units: Sequence[UnitSpec], weights: Dict[str, torch.Tensor],
             acts: Union[Dict[str, torch.Tensor], RowsFn], grads: Union[Dict[str, torch.Tensor], RowsFn, None],
             n_tokens: int, lam: float = 1e-2, budget: Optional[int] = None, fixed_rank: Optional[int] = None,
             mode: int = K.KF_KEY_HALF_SIGMA2, quant: bool = False, tol: float = 1e-6, max_sweeps: int = 30,
             stream=None, sync_timer: Optional[Callable[[str], None]] = None,
             site_dims: Optional[Dict[str, int]] = None, act_sites: Optional[Sequence[str]] = None,
             groups: Optional[Sequence[Sequence[int]]] = None, chunk_tokens: int = 16384,
             keep_covs: Union[bool, Sequence[str]] = True, keep_whitened: bool = True,
             score: Optional[str] = None, unit_weights: Optional[Sequence[float]] = None,
             defer_allocation: bool = False, alpha: Optional[float] = None) -> Result:
    """Runs the five steps.

    ``acts``/``grads``: dicts of resident (n_tokens x d) device tensors, or ``acts`` a callable
    ``rows(site, t0, t1)`` returning device rows of any site (``grads`` is then ignored), with
    ``site_dims`` giving every site's width and ``act_sites`` naming the activation sites (the
    ones fake-quantised when ``quant``).
    ``groups``: lists of unit indices processed one after the other (default: one group).
    ``keep_covs``: keep every finished covariance in the result (True), none (False) or the
    named sites only; ``keep_whitened=False`` releases W~ after its spectrum and, per unit,
    the factor that the unwhitening does not read.
    ``score``: "half_sigma2" (default; ``mode`` may also select the per-parameter key),
    "energy_ratio" (UniRank: sigma^2 / ||Sigma||^2 of the unit, times ``unit_weights``, its
    layer importance) or "empirical_fisher" (LASER: each component's contribution to the
    empirical-Fisher loss, 1/2 mean_t (a_t . u_i)^2 (g_t . v_i)^2, from a second pass over the
    calibration rows with every component mapped back; the kept set of a unit is then any
    subset, and its factors are the kept columns of U and rows of V), or "swift_hybrid"
    (Swift-SVD's hybrid score beta^alpha log(e + eps*_k)^(1 - alpha) per component, with
    ``unit_weights`` the layers' importance beta and ``alpha`` in [0, 1]).
    ``stream``: a torch.cuda.Stream or None; the whole driver runs on it.  Device-side
    failures (a non-positive Cholesky pivot, Jacobi not converged, a wait that gave up) are
    raised as KfsvdError at the host read of the ranks.
    ``defer_allocation``: stop after the spectra (steps 1-4) and return the units with their
    sigma, vecs and the factors the unwhitening reads (ranks, cut and used are None); the
    sharded driver allocates over every rank's spectra and then maps back with ``_finish``.
    ``sync_timer(tag)`` (optional) is called at phase boundaries ("kfac", "whiten", "svd",
    "allocate", "unwhiten"; per group for the first three; "score" after the empirical-Fisher
    pass) and around every kfac_accumulate and empirical_fisher_accumulate call ("syrk<",
    "syrk>", "fisher<", "fisher>"), so a caller can record CUDA events there.
    """
    if score not in SCORES:
        raise ValueError("compress: unknown score %r" % (score,))
    if score in ("energy_ratio", "empirical_fisher", "swift_hybrid") and (budget is None or fixed_rank is not None) \
            and not defer_allocation:
        raise ValueError("compress: score %r needs a budget and no fixed rank" % (score,))
    with _on_stream(stream):
        return _compress(ctx, units, weights, acts, grads, n_tokens, lam, budget, fixed_rank, mode, quant, tol,
                         max_sweeps, stream, sync_timer, site_dims, act_sites, groups, chunk_tokens, keep_covs,
                         keep_whitened, score, unit_weights, defer_allocation, alpha)


def _compress(ctx, units, weights, acts, grads, n_tokens, lam, budget, fixed_rank, mode, quant, tol, max_sweeps,
              stream, sync_timer, site_dims, act_sites, groups, chunk_tokens, keep_covs, keep_whitened, score,
              unit_weights, defer_allocation, alpha) -> Result:
    mark = sync_timer or (lambda _name: None)
    dev = next(iter(weights.values())).device
    if callable(acts):
        rows_fn = acts
        dims = dict(site_dims or {})
        quant_sites = set(act_sites or [])
    else:
        resident = dict(acts)
        resident.update(grads or {})
        rows_fn = lambda name, t0, t1: resident[name][t0:t1]
        dims = {k: v.shape[1] for k, v in resident.items()}
        quant_sites = set(acts.keys())
        chunk_tokens = max(n_tokens, 1)   # resident rows: one call per site
    groups = [list(range(len(units)))] if groups is None else [list(g) for g in groups]

    outs: List[Optional[UnitOut]] = [None] * len(units)
    sweeps_dev = torch.zeros(len(units), dtype=torch.int32, device=dev)
    all_covs: Dict[str, torch.Tensor] = {}
    for grp in groups:
        # ---- step 1: the group's calibration sites
        needed: List[str] = []
        for i in grp:
            for sname in (units[i].x_site, units[i].g_site):
                if sname not in needed:
                    needed.append(sname)
        covs: Dict[str, torch.Tensor] = {}
        for sname in needed:
            d = dims[sname]
            cov = torch.zeros((d, d), dtype=torch.float32, device=dev)
            q = K.KF_QUANT_INT8_TOKEN if (quant and sname in quant_sites) else K.KF_QUANT_NONE
            for t0 in range(0, n_tokens, chunk_tokens):
                rows = rows_fn(sname, t0, min(n_tokens, t0 + chunk_tokens))
                mark("syrk<")
                K.kfac_accumulate(ctx, rows, cov, quant=q, stream=stream)
                mark("syrk>")
                del rows
            K.kf_finalize_covariance(ctx, cov, n_tokens, lam, stream=stream)
            covs[sname] = cov
        mark("kfac")

        # ---- steps 2 and 3: factors and whitened weights (a factor is shared by the units
        # that use the same block of the same site)
        # step 2 for the whole group at once: every distinct factor (S_x = chol(X)^T per input
        # block, S_g = chol(G) per output block) and the Gram-side inverses, as independent
        # chains side by side (factor_covariances); the whiten calls below reuse them
        fx: Dict[tuple, torch.Tensor] = {}
        fg: Dict[tuple, torch.Tensor] = {}
        inv_x: Dict[tuple, torch.Tensor] = {}
        inv_g: Dict[tuple, torch.Tensor] = {}
        want_ix = {(units[i].x_site, units[i].x_off, units[i].m) for i in grp
                   if K.kf_gram_side(units[i].m, units[i].n) == K.KF_SIDE_LEFT}
        want_ig = {(units[i].g_site, units[i].g_off, units[i].n) for i in grp
                   if K.kf_gram_side(units[i].m, units[i].n) == K.KF_SIDE_RIGHT}
        jobs = []
        for i in grp:
            u = units[i]
            kx, kg = (u.x_site, u.x_off, u.m), (u.g_site, u.g_off, u.n)
            if kx not in fx:
                fx[kx] = torch.empty((u.m, u.m), dtype=torch.float32, device=dev)
                if kx in want_ix:
                    inv_x[kx] = torch.empty((u.m, u.m), dtype=torch.float32, device=dev)
                jobs.append((covs[u.x_site][u.x_off:u.x_off + u.m, u.x_off:u.x_off + u.m], fx[kx], inv_x.get(kx), True))
            if kg not in fg:
                fg[kg] = torch.empty((u.n, u.n), dtype=torch.float32, device=dev)
                if kg in want_ig:
                    inv_g[kg] = torch.empty((u.n, u.n), dtype=torch.float32, device=dev)
                jobs.append((covs[u.g_site][u.g_off:u.g_off + u.n, u.g_off:u.g_off + u.n], fg[kg], inv_g.get(kg), False))
        K.factor_covariances(ctx, jobs, stream=stream)
        del jobs
        # step 3: one workspace for the group's whiten calls; consecutive units that share a
        # factor (and a shape) reuse its bfloat16 planes from the previous call
        wws = torch.empty(max(K.whiten_workspace_size(units[i].m, units[i].n) for i in grp), dtype=torch.uint8,
                          device=dev)
        planes_of = None          # (m, n, x key, g key) of the planes left in wws
        for i in grp:
            u = units[i]
            side = K.kf_gram_side(u.m, u.n)
            kx, kg = (u.x_site, u.x_off, u.m), (u.g_site, u.g_off, u.n)
            flags = K.KF_REUSE_SX | K.KF_REUSE_SG | K.KF_REUSE_SINV
            Sx, Sg = fx[kx], fg[kg]
            Sinv = inv_x[kx] if side == K.KF_SIDE_LEFT else inv_g[kg]
            X = covs[u.x_site][u.x_off:u.x_off + u.m, u.x_off:u.x_off + u.m]
            G = covs[u.g_site][u.g_off:u.g_off + u.n, u.g_off:u.g_off + u.n]
            W = weights[u.weight][u.row0:u.row0 + u.m, u.col0:u.col0 + u.n]
            Wt = torch.empty((u.m, u.n), dtype=torch.float32, device=dev)
            if planes_of is not None and planes_of[:2] == (u.m, u.n):
                if planes_of[2] == kx:
                    flags |= K.KF_REUSE_SX_PLANES
                if planes_of[3] == kg:
                    flags |= K.KF_REUSE_SG_PLANES
            K.whiten(ctx, X, G, W, Sx, Sg, Sinv, Wt, flags=flags, workspace=wws, stream=stream)
            planes_of = (u.m, u.n, kx, kg)
            keep_x = keep_whitened or side == K.KF_SIDE_LEFT
            keep_g = keep_whitened or side == K.KF_SIDE_RIGHT
            outs[i] = UnitOut(u.name, u.m, u.n, side, Sx if keep_x else None, Sg if keep_g else None, Sinv, Wt)
        del fx, fg, inv_x, inv_g, wws
        if keep_covs is True:
            all_covs.update(covs)
        elif keep_covs:
            all_covs.update({k: v for k, v in covs.items() if k in set(keep_covs)})
        del covs
        mark("whiten")

        # ---- step 4: spectra, batched by min(m, n)
        by_s: Dict[int, List[int]] = {}
        for i in grp:
            by_s.setdefault(min(units[i].m, units[i].n), []).append(i)
        for s, idx in by_s.items():
            for i in idx:
                outs[i].sigma = torch.empty(s, dtype=torch.float32, device=dev)
                outs[i].vecs = torch.empty((s, s), dtype=torch.float32, device=dev)
            sw = torch.zeros(len(idx), dtype=torch.int32, device=dev)
            K.whitened_svd(ctx, [outs[i].Wt for i in idx], [outs[i].sigma for i in idx],
                           [outs[i].vecs for i in idx], sweeps=sw, tol=tol, max_sweeps=max_sweeps, stream=stream)
            sweeps_dev[torch.tensor(idx, device=dev)] = sw
            if not keep_whitened:
                for i in idx:
                    outs[i].Wt = None
        mark("svd")

    if defer_allocation:
        ctx.sync_status(stream)
        for o, sw_ in zip(outs, sweeps_dev.cpu().tolist()):
            o.sweeps = int(sw_)
        return Result(outs, all_covs, None, None, None)

    # ---- step 5a: global allocation
    sig = torch.cat([o.sigma for o in outs])
    lens = [min(o.m, o.n) for o in outs]
    off = torch.tensor([0] + list(_cumsum(lens)), dtype=torch.int64, device=dev)
    cost = torch.tensor([o.m + o.n for o in outs], dtype=torch.int64, device=dev)
    ranks = torch.empty(len(outs), dtype=torch.int32, device=dev)
    cut = torch.empty(2, dtype=torch.float32, device=dev)
    used = torch.zeros(1, dtype=torch.int64, device=dev)
    if score == "empirical_fisher":
        qsites = quant_sites if quant else set()
        return _fisher_allocation(ctx, units, outs, weights, rows_fn, qsites, n_tokens, chunk_tokens, int(budget),
                                  off, cost, ranks, cut, used, sweeps_dev, all_covs, stream, mark)
    _allocate(ctx, sig, off, cost, budget, ranks, cut, used, stream, score=score, mode=mode, fixed_rank=fixed_rank,
              unit_weights=unit_weights, alpha=alpha)
    return _finish(ctx, units, outs, weights, ranks, cut, used, sweeps_dev, all_covs, stream, mark)


def _finish(ctx, units, outs, weights, ranks, cut, used, sweeps_dev, all_covs, stream, mark) -> Result:
    dev = ranks.device
    ctx.sync_status(stream)
    ranks_h = ranks.cpu().tolist()
    sweeps_h = sweeps_dev.cpu().tolist()
    mark("allocate")

    # ---- step 5b: factors in the original space
    for o, u, r, sw in zip(outs, units, ranks_h, sweeps_h):
        o.rank = int(r)
        o.sweeps = int(sw)
        o.U = torch.empty((o.m, max(o.rank, 1)), dtype=torch.float32, device=dev)[:, :o.rank]
        o.V = torch.empty((max(o.rank, 1), o.n), dtype=torch.float32, device=dev)[:o.rank]
        if o.rank > 0:
            W = weights[u.weight][u.row0:u.row0 + u.m, u.col0:u.col0 + u.n]
            K.unwhiten(ctx, W, o.Sx, o.Sg, o.Sinv, o.sigma, o.vecs, o.rank, o.U, o.V, stream=stream)
    mark("unwhiten")
    return Result(outs, all_covs, ranks, cut, used)


def _fisher_allocation(ctx, units, outs, weights, rows_fn, quant_sites, n_tokens, chunk_tokens, budget, off, cost,
                       ranks, cut, used, sweeps_dev, all_covs, stream, mark) -> Result:
    """LASER's empirical-Fisher allocation: every component mapped back (U_all, V_all), its
    score accumulated over the calibration rows, then sort-and-truncate on the scores.  The
    activations of ``quant_sites`` are fake-quantised over their full width first, as they
    were for the covariance."""
    dev = ranks.device
    keys = []
    full = []
    for o, u in zip(outs, units):
        s = min(o.m, o.n)
        W = weights[u.weight][u.row0:u.row0 + u.m, u.col0:u.col0 + u.n]
        Ua = torch.empty((o.m, s), dtype=torch.float32, device=dev)
        Va = torch.empty((s, o.n), dtype=torch.float32, device=dev)
        K.unwhiten(ctx, W, o.Sx, o.Sg, o.Sinv, o.sigma, o.vecs, s, Ua, Va, stream=stream)
        acc = torch.zeros(s, dtype=torch.float64, device=dev)
        for t0 in range(0, n_tokens, chunk_tokens):
            t1 = min(n_tokens, t0 + chunk_tokens)
            a = rows_fn(u.x_site, t0, t1)
            if u.x_site in quant_sites:
                qa = torch.empty(a.shape, dtype=torch.bfloat16, device=dev)
                K.fake_quant_rows(ctx, a, qa, stream=stream)
                a = qa
            a = a[:, u.x_off:u.x_off + u.m]
            g = rows_fn(u.g_site, t0, t1)[:, u.g_off:u.g_off + u.n]
            mark("fisher<")
            K.empirical_fisher_accumulate(ctx, a, g, Ua, Va, acc, stream=stream)
            mark("fisher>")
        k_ = torch.empty(s, dtype=torch.float32, device=dev)
        K.empirical_fisher_finalize(ctx, acc, n_tokens, k_, stream=stream)
        keys.append(k_)
        full.append((Ua, Va))
    mark("score")
    keys_t = torch.cat(keys)
    keep = torch.empty(keys_t.numel(), dtype=torch.uint8, device=dev)
    K.score_and_allocate_keys(ctx, keys_t, off, cost, budget, ranks, keep=keep, cut=cut, used=used, stream=stream)
    ctx.sync_status(stream)
    ranks_h = ranks.cpu().tolist()
    sweeps_h = sweeps_dev.cpu().tolist()
    mark("allocate")
    offs = off.cpu().tolist()
    for i, (o, (Ua, Va), r, sw) in enumerate(zip(outs, full, ranks_h, sweeps_h)):
        o.rank = int(r)
        o.sweeps = int(sw)
        sel = K.compact_mask(ctx, keep[offs[i]:offs[i + 1]], 1, stream=stream)
        o.U = K.gather_rows_cols(ctx, Ua, col_idx=sel, stream=stream)
        o.V = K.gather_rows_cols(ctx, Va, row_idx=sel, stream=stream)
        o.kept = sel
        o.scores = keys[i]
    mark("unwhiten")
    return Result(outs, all_covs, ranks, cut, used)


@dataclass
class ActUnitOut:
    name: str
    m: int
    n: int
    C: Optional[torch.Tensor]            # n x n output covariance (released unless kept)
    sigma: Optional[torch.Tensor] = None  # n values, descending (sqrt of C's eigenvalues)
    vecs: Optional[torch.Tensor] = None   # n x n, eigenvectors as columns
    sweeps: int = 0
    rank: int = 0
    U: Optional[torch.Tensor] = None      # m x rank: W V_k
    V: Optional[torch.Tensor] = None      # rank x n: V_k^T


def compress_activation_only(ctx: K.Context, units: Sequence[UnitSpec], weights: Dict[str, torch.Tensor],
                             acts: Union[Dict[str, torch.Tensor], RowsFn], n_tokens: int, budget: int,
                             quant: bool = False, tol: float = 1e-6, max_sweeps: int = 30, stream=None,
                             sync_timer: Optional[Callable[[str], None]] = None,
                             site_dims: Optional[Dict[str, int]] = None,
                             groups: Optional[Sequence[Sequence[int]]] = None, chunk_tokens: int = 16384,
                             keep_cov: bool = False) -> Result:
    """Swift-SVD's activation-only route: W_k = W V_k V_k^T with V_k the top eigenvectors of
    the covariance of the layer output, C = (1/N) sum_t (a_t W)^T (a_t W); no gradients, no
    Cholesky.  Per group: the activation second moment of every input site (kfac_accumulate,
    fake-quantised rows when ``quant``; finalised without damping), C = W^T X W per unit
    (activation_covariance), the eigenpairs in batches of equal n (activation_eig); then one
    global sort-and-truncate on 1/2 sigma^2 over the first min(m, n) components of every
    unit (score_and_allocate) and the factors U = W V_k, V = V_k^T (activation_factors).
    ``acts``, ``groups`` and ``stream`` as for ``compress``; ``sync_timer`` tags: "kfac", "cov",
    "eig" per group, "allocate", "factors", and "syrk<"/"syrk>" around every kfac_accumulate."""
    with _on_stream(stream):
        return _compress_activation_only(ctx, units, weights, acts, n_tokens, budget, quant, tol, max_sweeps, stream,
                                         sync_timer, site_dims, groups, chunk_tokens, keep_cov)


def _compress_activation_only(ctx, units, weights, acts, n_tokens, budget, quant, tol, max_sweeps, stream, sync_timer,
                              site_dims, groups, chunk_tokens, keep_cov) -> Result:
    mark = sync_timer or (lambda _name: None)
    dev = next(iter(weights.values())).device
    if callable(acts):
        rows_fn = acts
        dims = dict(site_dims or {})
    else:
        resident = dict(acts)
        rows_fn = lambda name, t0, t1: resident[name][t0:t1]
        dims = {k: v.shape[1] for k, v in resident.items()}
        chunk_tokens = max(n_tokens, 1)
    groups = [list(range(len(units)))] if groups is None else [list(g) for g in groups]
    q = K.KF_QUANT_INT8_TOKEN if quant else K.KF_QUANT_NONE
    outs: List[Optional[ActUnitOut]] = [None] * len(units)
    sweeps_dev = torch.zeros(len(units), dtype=torch.int32, device=dev)
    for grp in groups:
        covs: Dict[str, torch.Tensor] = {}
        for i in grp:
            sname = units[i].x_site
            if sname in covs:
                continue
            d = dims[sname]
            cov = torch.zeros((d, d), dtype=torch.float32, device=dev)
            for t0 in range(0, n_tokens, chunk_tokens):
                rows = rows_fn(sname, t0, min(n_tokens, t0 + chunk_tokens))
                mark("syrk<")
                K.kfac_accumulate(ctx, rows, cov, quant=q, stream=stream)
                mark("syrk>")
                del rows
            K.kf_finalize_covariance(ctx, cov, n_tokens, 0.0, stream=stream)
            covs[sname] = cov
        mark("kfac")
        for i in grp:
            u = units[i]
            X = covs[u.x_site][u.x_off:u.x_off + u.m, u.x_off:u.x_off + u.m]
            W = weights[u.weight][u.row0:u.row0 + u.m, u.col0:u.col0 + u.n]
            C = torch.empty((u.n, u.n), dtype=torch.float32, device=dev)
            K.activation_covariance(ctx, X, W, C, stream=stream)
            outs[i] = ActUnitOut(u.name, u.m, u.n, C)
        del covs
        mark("cov")
        by_n: Dict[int, List[int]] = {}
        for i in grp:
            by_n.setdefault(units[i].n, []).append(i)
        for n, idx in by_n.items():
            for i in idx:
                outs[i].sigma = torch.empty(n, dtype=torch.float32, device=dev)
                outs[i].vecs = torch.empty((n, n), dtype=torch.float32, device=dev)
            sw = torch.zeros(len(idx), dtype=torch.int32, device=dev)
            K.activation_eig(ctx, [outs[i].C for i in idx], [outs[i].sigma for i in idx],
                             [outs[i].vecs for i in idx], sweeps=sw, tol=tol, max_sweeps=max_sweeps, stream=stream)
            sweeps_dev[torch.tensor(idx, device=dev)] = sw
            if not keep_cov:
                for i in idx:
                    outs[i].C = None
        mark("eig")

    lens = [min(o.m, o.n) for o in outs]
    sig = torch.cat([o.sigma[:s] for o, s in zip(outs, lens)])
    off = torch.tensor([0] + list(_cumsum(lens)), dtype=torch.int64, device=dev)
    cost = torch.tensor([o.m + o.n for o in outs], dtype=torch.int64, device=dev)
    ranks = torch.empty(len(outs), dtype=torch.int32, device=dev)
    cut = torch.empty(2, dtype=torch.float32, device=dev)
    used = torch.zeros(1, dtype=torch.int64, device=dev)
    K.score_and_allocate(ctx, sig, off, cost, int(budget), ranks, cut=cut, used=used, stream=stream)
    ctx.sync_status(stream)
    ranks_h = ranks.cpu().tolist()
    sweeps_h = sweeps_dev.cpu().tolist()
    mark("allocate")
    for o, u, r, swp in zip(outs, units, ranks_h, sweeps_h):
        o.rank = int(r)
        o.sweeps = int(swp)
        o.U = torch.empty((o.m, max(o.rank, 1)), dtype=torch.float32, device=dev)[:, :o.rank]
        o.V = torch.empty((max(o.rank, 1), o.n), dtype=torch.float32, device=dev)[:o.rank]
        if o.rank > 0:
            W = weights[u.weight][u.row0:u.row0 + u.m, u.col0:u.col0 + u.n]
            K.activation_factors(ctx, W, o.vecs, o.rank, o.U, o.V, stream=stream)
    mark("factors")
    return Result(outs, {}, ranks, cut, used)


def hybrid_ffn_split(ctx: K.Context, W_gate: torch.Tensor, W_up: torch.Tensor, X: torch.Tensor,
                     gate_factors, up_factors, n_svd: int, stream=None):
    """LASER's hybrid FFN channel selection for one FFN: the temporary factors (U, V) of gate
    and up (e.g. ``unwhiten`` at a temporary rank) score every hidden channel by the error of
    its pre-activation, d_j^T X d_j with d_j = (W - U V)[:, j], summed over gate and up; the
    f - n_svd channels with the largest error stay dense (equal errors keep the lower index
    dense) and the other n_svd are SVD-friendly.  Returns (svd_idx, dense_idx, errors, keys):
    increasing int64 channel indices, the float64 summed errors and their float32 keys."""
    dev = W_gate.device
    f = int(W_gate.shape[1])
    if not 0 <= n_svd <= f or int(W_up.shape[1]) != f:
        raise ValueError("hybrid_ffn_split: n_svd must lie in [0, d_ffn] and gate/up must share d_ffn")
    err = torch.zeros(f, dtype=torch.float64, device=dev)
    keys = torch.empty(f, dtype=torch.float32, device=dev)
    Ug, Vg = gate_factors
    Uu, Vu = up_factors
    K.channel_errors(ctx, W_gate, Ug, Vg, X, err, stream=stream)
    K.channel_errors(ctx, W_up, Uu, Vu, X, err, keys=keys, stream=stream)
    off = torch.tensor([0, f], dtype=torch.int64, device=dev)
    cost = torch.ones(1, dtype=torch.int64, device=dev)
    ranks = torch.empty(1, dtype=torch.int32, device=dev)
    keep = torch.empty(f, dtype=torch.uint8, device=dev)
    K.score_and_allocate_keys(ctx, keys, off, cost, f - n_svd, ranks, keep=keep, stream=stream)
    dense = K.compact_mask(ctx, keep, 1, stream=stream)
    svd = K.compact_mask(ctx, keep, 0, stream=stream)
    return svd, dense, err, keys


@dataclass
class HybridEntry:
    kind: str            # "unit": an ordinary unit; "svd": the SVD-friendly columns of a gate/up unit
    unit: int            # index into the caller's units
    out: UnitOut         # spectrum, rank and factors (for "svd": of W[:, svd_idx])
    svd_idx: Optional[torch.Tensor] = None


@dataclass
class HybridResult:
    entries: List[HybridEntry]
    splits: List[dict]   # per (gate, up) pair: "svd" and "dense" channel indices, "errors", "keys"
    ranks: torch.Tensor  # per entry
    cut: torch.Tensor
    used: torch.Tensor
    budget: int          # the budget left for the low-rank factors after the dense channels
    dense_cost: int


def compress_hybrid_ffn(ctx: K.Context, units: Sequence[UnitSpec], weights: Dict[str, torch.Tensor],
                        acts, grads, n_tokens: int, lam: float, budget: int, r_temp: int, n_svd: int,
                        pairs: Sequence[Sequence[int]], quant: bool = False, tol: float = 1e-6, max_sweeps: int = 30,
                        stream=None, site_dims: Optional[Dict[str, int]] = None,
                        act_sites: Optional[Sequence[str]] = None, chunk_tokens: int = 16384) -> HybridResult:
    """LASER's hybrid FFN inside the global allocation.  Steps 1-4 for every unit; for each
    (gate, up) pair of unit indices, the temporary factors at rank ``r_temp`` score the hidden
    channels (hybrid_ffn_split) and the ``n_svd`` SVD-friendly columns of gate and up are
    whitened again with their block G[S, S] of the gradient factor (gathered by index) and
    take part in the global allocation as units of their own; the other columns stay dense and
    their cost (d_model per channel and projection) is taken off the budget first.  Every
    other unit is allocated as usual; all entries are mapped back with ``unwhiten``."""
    with _on_stream(stream):
        return _compress_hybrid_ffn(ctx, units, weights, acts, grads, n_tokens, lam, budget, r_temp, n_svd, pairs,
                                    quant, tol, max_sweeps, stream, site_dims, act_sites, chunk_tokens)


def _compress_hybrid_ffn(ctx, units, weights, acts, grads, n_tokens, lam, budget, r_temp, n_svd, pairs, quant, tol,
                         max_sweeps, stream, site_dims, act_sites, chunk_tokens) -> HybridResult:
    keep = sorted({units[i].x_site for p in pairs for i in p} | {units[i].g_site for p in pairs for i in p})
    base = compress(ctx, units, weights, acts, grads, n_tokens, lam=lam, budget=None, quant=quant, tol=tol,
                    max_sweeps=max_sweeps, stream=stream, site_dims=site_dims, act_sites=act_sites,
                    chunk_tokens=chunk_tokens, keep_covs=keep, defer_allocation=True)
    outs = base.units
    dev = outs[0].sigma.device

    def wview(u: UnitSpec) -> torch.Tensor:
        return weights[u.weight][u.row0:u.row0 + u.m, u.col0:u.col0 + u.n]

    in_pair = {i for p in pairs for i in p}
    entries = [HybridEntry("unit", i, outs[i]) for i in range(len(units)) if i not in in_pair]
    w_of = {id(e.out): wview(units[e.unit]) for e in entries}
    splits = []
    dense_dm: List[int] = []     # per dense projection: d_model and its dense channel count
    dense_n: List[int] = []
    new_svd: List[HybridEntry] = []
    for gi, ui in pairs:
        facs = {}
        for i in (gi, ui):
            o, u = outs[i], units[i]
            U = torch.empty((u.m, max(r_temp, 1)), dtype=torch.float32, device=dev)[:, :r_temp]
            V = torch.empty((max(r_temp, 1), u.n), dtype=torch.float32, device=dev)[:r_temp]
            if r_temp > 0:
                K.unwhiten(ctx, wview(u), o.Sx, o.Sg, o.Sinv, o.sigma, o.vecs, r_temp, U, V, stream=stream)
            facs[i] = (U, V) if r_temp > 0 else (None, None)
        ug = units[gi]
        X = base.covs[ug.x_site][ug.x_off:ug.x_off + ug.m, ug.x_off:ug.x_off + ug.m]
        svd, dense, err, keys = hybrid_ffn_split(ctx, wview(ug), wview(units[ui]), X, facs[gi], facs[ui], n_svd,
                                                 stream=stream)
        splits.append({"gate": gi, "up": ui, "svd": svd, "dense": dense, "errors": err, "keys": keys})
        for i in (gi, ui):
            u = units[i]
            dense_dm.append(u.m)
            dense_n.append(int(dense.numel()))
            k = int(svd.numel())
            if k == 0:
                continue
            Xi = base.covs[u.x_site][u.x_off:u.x_off + u.m, u.x_off:u.x_off + u.m]
            Gi = base.covs[u.g_site][u.g_off:u.g_off + u.n, u.g_off:u.g_off + u.n]
            W_S = K.gather_rows_cols(ctx, wview(u), col_idx=svd, stream=stream)
            G_S = K.gather_rows_cols(ctx, Gi, row_idx=svd, col_idx=svd, stream=stream)
            s_ = min(u.m, k)
            Sx = torch.empty((u.m, u.m), dtype=torch.float32, device=dev)
            Sg = torch.empty((k, k), dtype=torch.float32, device=dev)
            Sinv = torch.empty((s_, s_), dtype=torch.float32, device=dev)
            Wt = torch.empty((u.m, k), dtype=torch.float32, device=dev)
            K.whiten(ctx, Xi, G_S, W_S, Sx, Sg, Sinv, Wt, stream=stream)
            e = HybridEntry("svd", i, UnitOut(u.name + ".svd", u.m, k, K.kf_gram_side(u.m, k), Sx, Sg, Sinv, Wt),
                            svd_idx=svd)
            w_of[id(e.out)] = W_S
            new_svd.append(e)
    by_s: Dict[int, List[HybridEntry]] = {}
    for e in new_svd:
        by_s.setdefault(min(e.out.m, e.out.n), []).append(e)
    for s_, grp in by_s.items():
        for e in grp:
            e.out.sigma = torch.empty(s_, dtype=torch.float32, device=dev)
            e.out.vecs = torch.empty((s_, s_), dtype=torch.float32, device=dev)
        sw = torch.zeros(len(grp), dtype=torch.int32, device=dev)
        K.whitened_svd(ctx, [e.out.Wt for e in grp], [e.out.sigma for e in grp], [e.out.vecs for e in grp],
                       sweeps=sw, tol=tol, max_sweeps=max_sweeps, stream=stream)
        for e, v in zip(grp, sw.cpu().tolist()):
            e.out.sweeps = int(v)
    entries += new_svd

    lens = [min(e.out.m, e.out.n) for e in entries]
    sig = torch.cat([e.out.sigma for e in entries])
    off = torch.tensor([0] + list(_cumsum(lens)), dtype=torch.int64, device=dev)
    cost = torch.tensor([e.out.m + e.out.n for e in entries], dtype=torch.int64, device=dev)
    ranks = torch.empty(len(entries), dtype=torch.int32, device=dev)
    cut = torch.empty(2, dtype=torch.float32, device=dev)
    used = torch.zeros(1, dtype=torch.int64, device=dev)
    left, dense_cost = K.kf_hybrid_ffn_budget(int(budget), dense_dm, dense_n, with_cost=True)
    K.score_and_allocate(ctx, sig, off, cost, left, ranks, cut=cut, used=used, stream=stream)
    ctx.sync_status(stream)
    for e, r in zip(entries, ranks.cpu().tolist()):
        o = e.out
        o.rank = int(r)
        o.U = torch.empty((o.m, max(o.rank, 1)), dtype=torch.float32, device=dev)[:, :o.rank]
        o.V = torch.empty((max(o.rank, 1), o.n), dtype=torch.float32, device=dev)[:o.rank]
        if o.rank > 0:
            K.unwhiten(ctx, w_of[id(o)], o.Sx, o.Sg, o.Sinv, o.sigma, o.vecs, o.rank, o.U, o.V, stream=stream)
    return HybridResult(entries, splits, ranks, cut, used, left, dense_cost)


def _cumsum(xs):
    t = 0
    for x in xs:
        t += x
        yield t
