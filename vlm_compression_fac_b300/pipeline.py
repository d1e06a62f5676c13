"""Whole-workload driver over the C ABI: the call a user makes to compress a set of layers.

For every calibration site it streams the rows into a K-FAC factor (kfac_accumulate) and
finalises it (kf_finalize_covariance); for every unit it whitens W (whiten, sharing the
input factor S_x between the units that read the same site); it takes the spectra of all
units in batches of equal min(m, n) (whitened_svd); it allocates ranks globally
(score_and_allocate) and maps the kept factors back (unwhiten).  The only host round trip
is reading the per-unit ranks after the allocation, to size U and V.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Callable, Dict, List, Optional, Sequence

import torch

from . import kfsvd as K


@dataclass
class UnitSpec:
    name: str
    m: int
    n: int
    x_site: str
    g_site: str


@dataclass
class UnitOut:
    name: str
    m: int
    n: int
    side: int
    Sx: torch.Tensor
    Sg: torch.Tensor
    Sinv: torch.Tensor
    Wt: torch.Tensor
    sigma: Optional[torch.Tensor] = None
    vecs: Optional[torch.Tensor] = None
    sweeps: int = 0
    rank: int = 0
    U: Optional[torch.Tensor] = None
    V: Optional[torch.Tensor] = None


@dataclass
class Result:
    units: List[UnitOut]
    covs: Dict[str, torch.Tensor]
    ranks: torch.Tensor
    cut: torch.Tensor
    used: torch.Tensor
    timings: Dict[str, float] = field(default_factory=dict)


def compress(ctx: K.Context, units: Sequence[UnitSpec], weights: Dict[str, torch.Tensor],
             acts: Dict[str, torch.Tensor], grads: Dict[str, torch.Tensor], n_tokens: int, lam: float = 1e-2,
             budget: Optional[int] = None, fixed_rank: Optional[int] = None, mode: int = K.KF_KEY_HALF_SIGMA2,
             quant: bool = False, tol: float = 1e-6, max_sweeps: int = 30, stream=None,
             sync_timer: Optional[Callable[[str], None]] = None) -> Result:
    """Runs the five steps on device-resident calibration rows and weights.

    ``sync_timer(tag)`` (optional) is called at phase boundaries ("kfac", "whiten", "svd",
    "allocate", "unwhiten") and around every kfac_accumulate call ("syrk<", "syrk>"), so a
    caller can record CUDA events there."""
    dev = next(iter(weights.values())).device
    mark = sync_timer or (lambda _name: None)

    covs: Dict[str, torch.Tensor] = {}
    for name, rows in list(acts.items()) + list(grads.items()):
        d = rows.shape[1]
        cov = torch.zeros((d, d), dtype=torch.float32, device=rows.device)
        q = K.KF_QUANT_INT8_TOKEN if (quant and name in acts) else K.KF_QUANT_NONE
        mark("syrk<")
        K.kfac_accumulate(ctx, rows, cov, quant=q, stream=stream)
        mark("syrk>")
        K.kf_finalize_covariance(ctx, cov, n_tokens, lam, stream=stream)
        covs[name] = cov
    mark("kfac")

    outs: List[UnitOut] = []
    sx_done: Dict[str, torch.Tensor] = {}
    sxinv_done: Dict[str, torch.Tensor] = {}
    for u in units:
        side = K.kf_gram_side(u.m, u.n)
        s = min(u.m, u.n)
        flags = 0
        if u.x_site in sx_done:
            Sx = sx_done[u.x_site]
            flags |= K.KF_REUSE_SX
        else:
            Sx = torch.empty((u.m, u.m), dtype=torch.float32, device=dev)
            sx_done[u.x_site] = Sx
        if side == K.KF_SIDE_LEFT:
            if u.x_site in sxinv_done:
                Sinv = sxinv_done[u.x_site]
                flags |= K.KF_REUSE_SINV
            else:
                Sinv = torch.empty((s, s), dtype=torch.float32, device=dev)
                sxinv_done[u.x_site] = Sinv
                flags &= ~K.KF_REUSE_SX  # the left inverse is computed together with S_x
        else:
            Sinv = torch.empty((s, s), dtype=torch.float32, device=dev)
        Sg = torch.empty((u.n, u.n), dtype=torch.float32, device=dev)
        Wt = torch.empty((u.m, u.n), dtype=torch.float32, device=dev)
        K.whiten(ctx, covs[u.x_site], covs[u.g_site], weights[u.name], Sx, Sg, Sinv, Wt, flags=flags,
                 stream=stream)
        outs.append(UnitOut(u.name, u.m, u.n, side, Sx, Sg, Sinv, Wt))
    mark("whiten")

    groups: Dict[int, List[int]] = {}
    for i, o in enumerate(outs):
        groups.setdefault(min(o.m, o.n), []).append(i)
    sweeps_all = torch.zeros(len(outs), dtype=torch.int32, device=dev)
    for s, idx in groups.items():
        for i in idx:
            outs[i].sigma = torch.empty(s, dtype=torch.float32, device=dev)
            outs[i].vecs = torch.empty((s, s), dtype=torch.float32, device=dev)
        sw = torch.zeros(len(idx), dtype=torch.int32, device=dev)
        K.whitened_svd(ctx, [outs[i].Wt for i in idx], [outs[i].sigma for i in idx], [outs[i].vecs for i in idx],
                       sweeps=sw, tol=tol, max_sweeps=max_sweeps, stream=stream)
        sweeps_all[torch.tensor(idx, device=dev)] = sw
    mark("svd")

    sig = torch.cat([o.sigma for o in outs])
    lens = [min(o.m, o.n) for o in outs]
    off = torch.tensor([0] + list(_cumsum(lens)), dtype=torch.int64, device=dev)
    cost = torch.tensor([o.m + o.n for o in outs], dtype=torch.int64, device=dev)
    ranks = torch.empty(len(outs), dtype=torch.int32, device=dev)
    cut = torch.empty(2, dtype=torch.float32, device=dev)
    used = torch.zeros(1, dtype=torch.int64, device=dev)
    if fixed_rank is not None:
        fr = torch.full((len(outs),), int(fixed_rank), dtype=torch.int32, device=dev)
        K.score_and_allocate(ctx, sig, off, cost, 0, ranks, mode=K.KF_FIXED_RANK, fixed_rank=fr, cut=cut,
                             used=used, stream=stream)
    else:
        K.score_and_allocate(ctx, sig, off, cost, int(budget), ranks, mode=mode, cut=cut, used=used,
                             stream=stream)
    ranks_h = ranks.cpu().tolist()
    sweeps_h = sweeps_all.cpu().tolist()
    mark("allocate")

    for o, r, sw in zip(outs, ranks_h, sweeps_h):
        o.rank = int(r)
        o.sweeps = int(sw)
        o.U = torch.empty((o.m, max(o.rank, 1)), dtype=torch.float32, device=dev)[:, :o.rank]
        o.V = torch.empty((max(o.rank, 1), o.n), dtype=torch.float32, device=dev)[:o.rank]
        if o.rank > 0:
            K.unwhiten(ctx, weights[o.name], o.Sx, o.Sg, o.Sinv, o.sigma, o.vecs, o.rank, o.U, o.V, stream=stream)
    mark("unwhiten")
    return Result(outs, covs, ranks, cut, used)


def _cumsum(xs):
    t = 0
    for x in xs:
        t += x
        yield t
