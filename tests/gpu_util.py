"""Helpers shared by the GPU parity tests (no method arithmetic here)."""
import numpy as np


def rel_fro(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def lower(a):
    return np.tril(np.asarray(a, dtype=np.float64))


def to_dev(x, torch, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(x))
    if dtype is not None:
        t = t.to(dtype)
    return t.cuda()


def bf16_dev(x, torch):
    """float32 values that are exactly bfloat16 -> a bfloat16 device tensor (exact)."""
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16).cuda()


def host_weight(wl, unit, torch, cache=None):
    """The unit's weight block (m x n) with exactly the values of the host generator
    (recipes.gen_weight), produced by the generator's bit-identical device twin
    (test_device_generator_matches_host) and copied back: the numpy generator needs minutes
    for the full-size 70B and VLM weights.  Heads of one matrix share its cached copy."""
    from synth import device
    key = unit.weight
    full = cache.get(key) if cache is not None else None
    if full is None:
        full = device.weight_on_device(wl, unit, torch).float().cpu().numpy()
        if cache is not None and tuple(unit.weight_shape) != (unit.m, unit.n):
            cache[key] = full
    return np.ascontiguousarray(full[unit.row0:unit.row0 + unit.m, unit.col0:unit.col0 + unit.n])


def moved_components(ranks_gpu, alloc_oracle, sig_oracle):
    """Components on which the GPU's and the oracle's ranks disagree, as
    (unit, component index, relative distance of its oracle score from the oracle's cut)."""
    cut = alloc_oracle.cut_score if np.isfinite(alloc_oracle.cut_score) else alloc_oracle.next_score
    out = []
    for u, (rg, ro) in enumerate(zip(ranks_gpu, alloc_oracle.ranks)):
        rg, ro = int(rg), int(ro)
        for i in range(min(rg, ro), max(rg, ro)):
            sc = 0.5 * float(sig_oracle[u][i]) ** 2
            out.append((u, i, abs(sc - cut) / abs(cut)))
    return out


def rank_parity(ranks_gpu, alloc_oracle, sig_oracle, tie_rel):
    """Ranks equal except where every differing component has an oracle score within
    tie_rel (relative) of the oracle's cut score.  Returns (ok, moved components)."""
    mv = moved_components(ranks_gpu, alloc_oracle, sig_oracle)
    return all(d <= tie_rel for _, _, d in mv), mv
