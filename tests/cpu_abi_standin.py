"""A CPU stand-in for the libkfsvd calls, built from the fp64 oracle, for testing the Python
glue of ``vlm_compression_fac_b300.pipeline`` (index bookkeeping, budget accounting, the
order of the calls) without a GPU.

TEST INFRASTRUCTURE ONLY: it is installed with ``install(monkeypatch)`` inside a test, which
replaces the binding's functions for that test alone.  The package itself has no CPU path and
never imports this module.
"""
import numpy as np
import torch

import oracle as O


class _Ctx:
    def sync_status(self, *a, **k):
        return 0

    def close(self):
        pass


def _np(t):
    return t.detach().to(torch.float64).cpu().numpy()


def _put(dst, arr):
    dst.copy_(torch.from_numpy(np.ascontiguousarray(arr)).to(dst.dtype))


def kf_gram_side(m, n):
    return 0 if n <= m else 1


def kfac_accumulate(ctx, rows, cov, quant=0, workspace=None, stream=None):
    A = _np(rows)
    if quant:
        A = O.fake_quant_int8_token(A.astype(np.float32)).astype(np.float64)
    S = np.tril(O.covariance_sum(A))
    _put(cov, np.tril(_np(cov)) + S)


def kf_finalize_covariance(ctx, cov, n_tokens, lam, stream=None):
    L = np.tril(_np(cov))
    _put(cov, O.finalize_covariance(L + np.tril(L, -1).T, n_tokens, lam))


def whiten(ctx, X, G, W, Sx, Sg, Sinv, Wt, flags=0, workspace=None, stream=None):
    # like the library: factors (and the Gram-side inverse) flagged as present are reused
    m, n = W.shape
    sx, sg = O.cholesky_factors(_np(X), _np(G))
    if flags & 1:
        sx = _np(Sx)
    else:
        _put(Sx, sx)
    if flags & 2:
        sg = _np(Sg)
    else:
        _put(Sg, sg)
    if not flags & 4:
        _put(Sinv, np.linalg.inv(sg) if kf_gram_side(m, n) == 0 else np.linalg.inv(sx))
    _put(Wt, O.whiten(_np(W), sx, sg))


def factor_covariances(ctx, jobs, workspace=None, stream=None):
    for A, S, Sinv, upper in jobs:
        L = np.linalg.cholesky(_np(A))
        F = L.T.copy() if upper else L
        _put(S, F)
        if Sinv is not None:
            _put(Sinv, np.linalg.inv(F))


def whitened_svd(ctx, Wts, sigmas, vecs, sweeps=None, tol=1e-6, max_sweeps=30, workspace=None, stream=None):
    for i, (Wt, sg, V) in enumerate(zip(Wts, sigmas, vecs)):
        m, n = Wt.shape
        u, s, vt = np.linalg.svd(_np(Wt), full_matrices=False)
        _put(sg, s)
        _put(V, vt.T if kf_gram_side(m, n) == 0 else u)
        if sweeps is not None:
            sweeps[i] = 1


def _segments(t, off):
    o = off.cpu().tolist()
    a = t.detach().cpu().numpy()
    return [a[o[u]:o[u + 1]] for u in range(len(o) - 1)]


def score_and_allocate(ctx, sigma, seg_offset, cost, budget, ranks, mode=0, fixed_rank=None, cut=None, used=None,
                       workspace=None, stream=None):
    segs = _segments(sigma, seg_offset)
    costs = cost.cpu().tolist()
    if mode == 2:
        al = O.allocate(segs, costs, 0, O.FIXED_RANK, fixed_rank.cpu().tolist())
    else:
        key = {0: O.KEY_HALF_SIGMA2, 1: O.KEY_PER_PARAM, 3: O.KEY_ENERGY_RATIO}[mode]
        al = O.allocate(segs, costs, int(budget), key, precision="f32")
    ranks.copy_(torch.tensor(al.ranks, dtype=torch.int32))
    if used is not None:
        used.fill_(int(al.used))
    if cut is not None:
        cut.copy_(torch.tensor([al.cut_score, al.next_score], dtype=torch.float32))


def _put_alloc(al, ranks, cut, used):
    ranks.copy_(torch.tensor(al.ranks, dtype=torch.int32))
    if used is not None:
        used.fill_(int(al.used))
    if cut is not None:
        cut.copy_(torch.tensor([al.cut_score, al.next_score], dtype=torch.float32))


def score_and_allocate_weighted(ctx, sigma, seg_offset, cost, budget, ranks, mode=3, unit_weight=None, cut=None,
                                used=None, workspace=None, stream=None):
    segs = _segments(sigma, seg_offset)
    key = {0: O.KEY_HALF_SIGMA2, 1: O.KEY_PER_PARAM, 3: O.KEY_ENERGY_RATIO}[mode]
    w = None if unit_weight is None else unit_weight.cpu().tolist()
    _put_alloc(O.allocate(segs, cost.cpu().tolist(), int(budget), key, precision="f32", weights=w), ranks, cut, used)


def score_and_allocate_hybrid(ctx, sigma, seg_offset, cost, budget, ranks, alpha, importance=None, cut=None,
                              used=None, workspace=None, stream=None):
    segs = _segments(sigma, seg_offset)
    b = [1.0] * len(segs) if importance is None else importance.cpu().tolist()
    _put_alloc(O.allocate_swift_hybrid(segs, cost.cpu().tolist(), int(budget), b, alpha), ranks, cut, used)


def score_and_allocate_keys(ctx, keys, seg_offset, cost, budget, ranks, keep=None, cut=None, used=None,
                            workspace=None, stream=None):
    segs = [np.maximum(s.astype(np.float32), 0) for s in _segments(keys, seg_offset)]
    al = O.allocate_keys(segs, cost.cpu().tolist(), int(budget))
    ranks.copy_(torch.tensor(al.ranks, dtype=torch.int32))
    if keep is not None:
        o = seg_offset.cpu().tolist()
        mask = np.zeros(keep.numel(), np.uint8)
        n_keep = int(al.ranks.sum())
        mask[np.asarray(o)[al.order_unit[:n_keep]] + al.order_comp[:n_keep]] = 1
        keep.copy_(torch.from_numpy(mask))
    if used is not None:
        used.fill_(int(al.used))
    if cut is not None:
        cut.copy_(torch.tensor([al.cut_score, al.next_score], dtype=torch.float32))


def unwhiten(ctx, W, Sx, Sg, Sinv, sigma, vecs, r, U, V, workspace=None, stream=None):
    # Like the library, reads only the Gram-side factor and its inverse (the other factor may
    # have been released): right side U = W S_g V~_r, V = V~_r^T S_g^-1; left side
    # U = S_x^-1 U~_r Sigma_r, V = Sigma_r^-1 U~_r^T S_x W.
    if r == 0:
        return
    m, n = W.shape
    Wd = _np(W)
    s = _np(sigma)[:r]
    Q = _np(vecs)[:, :r]
    inv = _np(Sinv)
    if kf_gram_side(m, n) == 0:
        sg = _np(Sg)
        u_, v_ = Wd @ sg @ Q, Q.T @ inv
    else:
        sx = _np(Sx)
        u_, v_ = inv @ (Q * s[None, :]), (Q.T @ sx @ Wd) / s[:, None]
    _put(U, u_)
    _put(V, v_)


def channel_errors(ctx, W, U, V, X, err_sum, keys=None, workspace=None, stream=None):
    m, n = W.shape
    Uh = np.zeros((m, 0)) if U is None else _np(U)
    Vh = np.zeros((0, n)) if V is None else _np(V)
    e = _np(err_sum) + O.channel_errors(_np(W), Uh, Vh, _np(X))
    _put(err_sum, e)
    if keys is not None:
        _put(keys, e.astype(np.float32))


def compact_mask(ctx, mask, want=1, stream=None):
    m = mask.detach().cpu().numpy() != 0
    return torch.from_numpy(np.nonzero(m == bool(want))[0].astype(np.int64))


def gather_rows_cols(ctx, src, row_idx=None, col_idx=None, out=None, stream=None):
    t = src
    if row_idx is not None:
        t = t[row_idx]
    if col_idx is not None:
        t = t[:, col_idx]
    return t.contiguous().clone()


def fake_quant_rows(ctx, rows, out, stream=None):
    _put(out, O.fake_quant_int8_token(_np(rows).astype(np.float32)))


def empirical_fisher_accumulate(ctx, act, grad, U, V, score_sum, workspace=None, stream=None):
    A, G = _np(act), _np(grad)
    P = A @ _np(U)
    Q = G @ _np(V).T
    _put(score_sum, _np(score_sum) + np.sum(P * P * Q * Q, axis=0))


def empirical_fisher_finalize(ctx, score_sum, n_tokens, keys, stream=None):
    _put(keys, (_np(score_sum) / (2.0 * n_tokens)).astype(np.float32))


def activation_covariance(ctx, X, W, C, workspace=None, stream=None):
    Wd = _np(W)
    _put(C, Wd.T @ _np(X) @ Wd)


def activation_eig(ctx, Cs, sigmas, vecs, sweeps=None, tol=1e-6, max_sweeps=30, workspace=None, stream=None):
    for i, (C, sg, V) in enumerate(zip(Cs, sigmas, vecs)):
        s, Q = O.output_eig(_np(C))
        _put(sg, s)
        _put(V, Q)
        if sweeps is not None:
            sweeps[i] = 1


def activation_factors(ctx, W, vecs, r, U, V, workspace=None, stream=None):
    if r == 0:
        return
    u_, v_ = O.activation_factors(_np(W), _np(vecs), r)
    _put(U, u_)
    _put(V, v_)


NAMES = ["factor_covariances", "fake_quant_rows", "empirical_fisher_accumulate", "empirical_fisher_finalize", "activation_covariance", "activation_eig",
         "activation_factors", "kf_gram_side", "kfac_accumulate", "kf_finalize_covariance", "whiten",
         "whitened_svd", "score_and_allocate", "score_and_allocate_keys", "score_and_allocate_weighted",
         "score_and_allocate_hybrid", "unwhiten", "channel_errors",
         "compact_mask", "gather_rows_cols"]


def install(monkeypatch):
    """Replaces the binding's calls used by the pipeline with the stand-ins (this test only)."""
    from vlm_compression_fac_b300 import kfsvd
    g = globals()
    for name in NAMES:
        monkeypatch.setattr(kfsvd, name, g[name])
    return _Ctx()
