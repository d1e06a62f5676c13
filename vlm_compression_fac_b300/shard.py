"""Sharding the path across ranks (one process per GPU) by unit.

Steps 1-4 of every unit are independent, so each rank takes a share of the units chosen by
longest-processing-time order on their estimated work; the one exchange is an all-gather of
the per-unit float32 spectra (a few MB), after which every rank runs the identical,
deterministic global allocation (bit-identical ranks everywhere) and maps back its own units.
"""
from __future__ import annotations

from typing import Dict, List, Optional, Sequence

import torch
import torch.distributed as dist


def unit_work(m: int, n: int, n_tokens: int, sweeps: int = 16) -> float:
    """Estimated flops of one unit: its two covariance SYRKs (N d^2 / 2 each, counted per unit
    although units may share a site), the whitening products, the Gram and about 6 s^3 per
    Jacobi sweep."""
    s = min(m, n)
    return n_tokens * (m * m + n * n) / 2.0 + 2.0 * m * n * (m + n) + 2.0 * s * s * max(m, n) + 6.0 * sweeps * s ** 3


def lpt_partition(work: Sequence[float], world: int) -> List[List[int]]:
    """Longest-processing-time partition: units by decreasing work (ties: lower index first),
    each to the rank with the least work so far (ties: lower rank).  Every rank's list is
    returned in increasing unit order; the result depends only on (work, world)."""
    if world < 1:
        raise ValueError("lpt_partition: world must be >= 1")
    order = sorted(range(len(work)), key=lambda i: (-float(work[i]), i))
    loads = [0.0] * world
    parts: List[List[int]] = [[] for _ in range(world)]
    for i in order:
        r = min(range(world), key=lambda k: (loads[k], k))
        parts[r].append(i)
        loads[r] += float(work[i])
    return [sorted(p) for p in parts]


def gather_spectra(local: Dict[int, torch.Tensor], lens: Sequence[int], parts: Sequence[Sequence[int]],
                   group=None, device=None) -> torch.Tensor:
    """All-gathers the spectra of every rank's units and returns them concatenated in global
    unit order (unit u's segment at sum(lens[:u])).  ``local`` maps each of this rank's units
    (parts[rank]) to its float32 spectrum of length lens[u].  One all-gather of equal-sized
    packed buffers; the packing follows ``parts``, which every rank holds identically."""
    world = dist.get_world_size(group)
    rank = dist.get_rank(group)
    if len(parts) != world:
        raise ValueError("gather_spectra: one part per rank expected")
    mine = list(parts[rank])
    if sorted(local.keys()) != sorted(mine):
        raise ValueError("gather_spectra: local spectra do not match this rank's units")
    sizes = [sum(int(lens[u]) for u in p) for p in parts]
    L = max(max(sizes), 1)
    if device is not None:
        dev = torch.device(device)
    else:
        dev = next(iter(local.values())).device if local else torch.device("cpu")
    buf = torch.zeros(L, dtype=torch.float32, device=dev)
    pos = 0
    for u in mine:
        seg = local[u].reshape(-1)
        if seg.numel() != int(lens[u]):
            raise ValueError("gather_spectra: unit %d has %d values, expected %d" % (u, seg.numel(), lens[u]))
        buf[pos:pos + seg.numel()] = seg.to(torch.float32)
        pos += seg.numel()
    outs = [torch.empty(L, dtype=torch.float32, device=dev) for _ in range(world)]
    dist.all_gather(outs, buf, group=group)
    offs = [0]
    for ln in lens:
        offs.append(offs[-1] + int(ln))
    full = torch.empty(offs[-1], dtype=torch.float32, device=dev)
    for r in range(world):
        pos = 0
        for u in parts[r]:
            full[offs[u]:offs[u] + int(lens[u])] = outs[r][pos:pos + int(lens[u])]
            pos += int(lens[u])
    return full


def compress_sharded(ctx, units, weights, acts, grads, n_tokens: int, lam: float, budget: Optional[int],
                     group=None, work: Optional[Sequence[float]] = None, score: Optional[str] = None,
                     mode: Optional[int] = None, fixed_rank: Optional[int] = None,
                     unit_weights: Optional[Sequence[float]] = None, alpha: Optional[float] = None, **kw):
    """The whole path over all ranks of ``group``: this rank runs steps 1-4 for its share of the
    units (``pipeline.compress`` with the allocation deferred), the spectra are all-gathered,
    every rank runs the same allocation over all units, and each maps back its own units.
    The allocation options are those of ``pipeline.compress`` and mean the same here:
    ``score`` (1/2 sigma^2, "energy_ratio" or "swift_hybrid"), ``mode`` (the per-parameter
    key), ``fixed_rank``, ``unit_weights`` (one per unit of ``units``, global order) and
    ``alpha``.  LASER's empirical-Fisher score needs a second pass over every unit's rows
    before the global sort and is not offered here (ValueError).  Any other keyword goes to
    ``pipeline.compress`` for steps 1-4.
    Returns (this rank's unit indices, their pipeline.UnitOut, the global ranks tensor,
    cut, used)."""
    from . import kfsvd as K
    from . import pipeline
    if score not in (None, "half_sigma2", "energy_ratio", "swift_hybrid"):
        raise ValueError("compress_sharded: score %r is not supported across ranks" % (score,))
    if unit_weights is not None and len(unit_weights) != len(units):
        raise ValueError("compress_sharded: unit_weights needs one weight per unit")
    if (budget is None) == (fixed_rank is None) or (fixed_rank is not None and score not in (None, "half_sigma2")):
        raise ValueError("compress_sharded: give a budget or a fixed rank (the latter with the default score)")
    world = dist.get_world_size(group)
    rank = dist.get_rank(group)
    w = list(work) if work is not None else [unit_work(u.m, u.n, n_tokens) for u in units]
    parts = lpt_partition(w, world)
    mine = parts[rank]
    outs = pipeline.compress(ctx, [units[i] for i in mine], weights, acts, grads, n_tokens, lam=lam,
                             budget=None, defer_allocation=True, **kw)
    lens = [min(u.m, u.n) for u in units]
    full = gather_spectra({i: o.sigma for i, o in zip(mine, outs.units)}, lens, parts, group,
                          device=next(iter(weights.values())).device)
    dev = full.device
    off = torch.tensor([0] + list(pipeline._cumsum(lens)), dtype=torch.int64, device=dev)
    cost = torch.tensor([u.m + u.n for u in units], dtype=torch.int64, device=dev)
    ranks = torch.empty(len(units), dtype=torch.int32, device=dev)
    cut = torch.empty(2, dtype=torch.float32, device=dev)
    used = torch.zeros(1, dtype=torch.int64, device=dev)
    pipeline._allocate(ctx, full, off, cost, 0 if budget is None else int(budget), ranks, cut, used, None,
                       score=score, mode=K.KF_KEY_HALF_SIGMA2 if mode is None else int(mode), fixed_rank=fixed_rank,
                       unit_weights=unit_weights, alpha=alpha)
    local_ranks = ranks[torch.tensor(mine, dtype=torch.int64, device=dev)] if mine else ranks[:0]
    sweeps = torch.tensor([o.sweeps for o in outs.units], dtype=torch.int32, device=dev)
    res = pipeline._finish(ctx, [units[i] for i in mine], outs.units, weights, local_ranks, cut, used, sweeps, {},
                           None, lambda _t: None)
    return mine, res.units, ranks, cut, used
