"""Thin ctypes binding of libkfsvd.so (include/kfsvd.h): argument marshalling only.

Every function has the name of the C entry point it calls and takes torch tensors for the
device buffers (PyTorch provides device memory and streams; every step of the path runs in
the library's CUDA kernels).  Workspace tensors are allocated here with torch when the
caller does not pass one.  A non-OK status raises KfsvdError.  There is no fallback: if the
shared library is missing the import fails.
"""
from __future__ import annotations

import ctypes
import os
from typing import List, Optional, Sequence

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libkfsvd.so")

KF_OK, KF_ERR_INVALID, KF_ERR_WORKSPACE, KF_ERR_CUDA = 0, 1, 2, 3
KF_ERR_NOT_SPD, KF_ERR_NO_CONVERGENCE, KF_ERR_TIMEOUT, KF_ERR_UNSUPPORTED = 4, 5, 6, 7
KF_BF16, KF_F32 = 0, 1
KF_QUANT_NONE, KF_QUANT_INT8_TOKEN = 0, 1
KF_KEY_HALF_SIGMA2, KF_KEY_PER_PARAM, KF_FIXED_RANK, KF_KEY_ENERGY_RATIO = 0, 1, 2, 3
KF_SIDE_RIGHT, KF_SIDE_LEFT = 0, 1
KF_REUSE_SX, KF_REUSE_SG, KF_REUSE_SINV = 1, 2, 4
KF_REUSE_SX_PLANES, KF_REUSE_SG_PLANES = 8, 16

STATUS_NAMES = {0: "KF_OK", 1: "KF_ERR_INVALID", 2: "KF_ERR_WORKSPACE", 3: "KF_ERR_CUDA",
                4: "KF_ERR_NOT_SPD", 5: "KF_ERR_NO_CONVERGENCE", 6: "KF_ERR_TIMEOUT",
                7: "KF_ERR_UNSUPPORTED"}

EXPORTED = ["kf_create", "kf_destroy", "kf_last_error", "kf_launch_count", "kf_sync_status", "kf_gram_side",
            "kfac_accumulate_workspace_size", "kfac_accumulate", "fake_quant_rows", "kf_finalize_covariance",
            "whiten_workspace_size", "whiten", "kf_svd_profile_enable", "kf_svd_profile_read",
            "whitened_svd_workspace_size", "whitened_svd",
            "score_and_allocate_workspace_size", "score_and_allocate", "score_and_allocate_weighted",
            "score_and_allocate_keys", "score_and_allocate_noalloc", "score_and_allocate_hybrid",
            "kf_set_wait_limit", "kf_hybrid_ffn_budget", "kf_fp32_fma_probe",
            "factor_covariances_workspace_size", "factor_covariances",
            "empirical_fisher_workspace_size", "empirical_fisher_accumulate", "empirical_fisher_finalize",
            "unwhiten_workspace_size", "unwhiten",
            "activation_covariance_workspace_size", "activation_covariance", "activation_eig_workspace_size",
            "activation_eig", "activation_factors_workspace_size", "activation_factors",
            "channel_errors_workspace_size", "channel_errors", "gather_rows_cols", "compact_mask"]


class KfsvdError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__("%s: %s" % (STATUS_NAMES.get(status, str(status)), msg))
        self.status = status


class SvdProblem(ctypes.Structure):
    _fields_ = [("Wt", ctypes.c_void_p), ("m", ctypes.c_int64), ("n", ctypes.c_int64),
                ("ldw", ctypes.c_int64), ("sigma", ctypes.c_void_p), ("vecs", ctypes.c_void_p),
                ("ldv", ctypes.c_int64), ("sweeps", ctypes.c_void_p)]


class SymProblem(ctypes.Structure):
    _fields_ = [("C", ctypes.c_void_p), ("n", ctypes.c_int64), ("ldc", ctypes.c_int64),
                ("sigma", ctypes.c_void_p), ("vecs", ctypes.c_void_p), ("ldv", ctypes.c_int64),
                ("sweeps", ctypes.c_void_p)]


class FactorJob(ctypes.Structure):
    _fields_ = [("A", ctypes.c_void_p), ("lda", ctypes.c_int64), ("n", ctypes.c_int64), ("S", ctypes.c_void_p),
                ("lds", ctypes.c_int64), ("Sinv", ctypes.c_void_p), ("ldsi", ctypes.c_int64),
                ("upper", ctypes.c_int32)]


class SvdProfile(ctypes.Structure):
    _fields_ = [("gram_ms", ctypes.c_float), ("jacobi_ms", ctypes.c_float), ("rayleigh_ms", ctypes.c_float),
                ("refine_ms", ctypes.c_float), ("jacobi_steps", ctypes.c_int64),
                ("jacobi_apply_flops", ctypes.c_double), ("jacobi_solve_ms", ctypes.c_float),
                ("jacobi_apply_ms", ctypes.c_float), ("jacobi_apply_launches", ctypes.c_int64),
                ("jacobi_apply_bytes", ctypes.c_double)]


_P, _I64, _I32, _U32, _F, _SZ = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_uint32,
                                 ctypes.c_float, ctypes.c_size_t)
_SIGS = {
    "kf_create": (_I32, [ctypes.c_int, ctypes.POINTER(ctypes.c_void_p)]),
    "kf_destroy": (None, [_P]),
    "kf_last_error": (ctypes.c_char_p, []),
    "kf_launch_count": (ctypes.c_uint64, []),
    "kf_sync_status": (_I32, [_P, _P, ctypes.POINTER(ctypes.c_int32)]),
    "kf_gram_side": (_I32, [_I64, _I64]),
    "kfac_accumulate_workspace_size": (_SZ, [_I32, _I32, _I64]),
    "kfac_accumulate": (_I32, [_P, _P, _I32, _I64, _I64, _I64, _I32, _P, _I64, _P, _SZ, _P]),
    "fake_quant_rows": (_I32, [_P, _P, _I32, _I64, _I64, _I64, _P, _P]),
    "kf_finalize_covariance": (_I32, [_P, _P, _I64, _I64, _I64, _F, _P]),
    "whiten_workspace_size": (_SZ, [_I64, _I64]),
    "whiten": (_I32, [_P, _P, _I64, _I64, _P, _I64, _I64, _P, _I32, _I64, _U32, _P, _I64, _P, _I64,
                      _P, _I64, _P, _I64, _P, _SZ, _P]),
    "kf_svd_profile_enable": (_I32, [_P, ctypes.c_int]),
    "kf_svd_profile_read": (_I32, [_P, ctypes.POINTER(SvdProfile)]),
    "whitened_svd_workspace_size": (_SZ, [_I32, _I64, _I64, _I64]),
    "whitened_svd": (_I32, [_P, _I32, ctypes.POINTER(SvdProblem), _F, _I32, _P, _SZ, _P]),
    "score_and_allocate_workspace_size": (_SZ, [_I64, _I32]),
    "score_and_allocate": (_I32, [_P, _P, _P, _P, _I32, _I64, _I64, _I32, _P, _P, _P, _P, _P, _SZ, _P]),
    "score_and_allocate_weighted": (_I32, [_P, _P, _P, _P, _I32, _I64, _I64, _I32, _P, _P, _P, _P, _P, _SZ, _P]),
    "score_and_allocate_keys": (_I32, [_P, _P, _P, _P, _I32, _I64, _I64, _P, _P, _P, _P, _P, _SZ, _P]),
    "score_and_allocate_noalloc": (_I32, [_P, _P, _P, _P, _I32, _I64, _I64, _I32, _P, _P, _P, _P, _P]),
    "score_and_allocate_hybrid": (_I32, [_P, _P, _P, _P, _I32, _I64, _I64, _P, ctypes.c_double, _P, _P, _P, _P,
                                         _SZ, _P]),
    "kf_set_wait_limit": (_I32, [_P, ctypes.c_uint64]),
    "factor_covariances_workspace_size": (_SZ, [_I32, ctypes.POINTER(FactorJob)]),
    "factor_covariances": (_I32, [_P, _I32, ctypes.POINTER(FactorJob), _P, _SZ, _P]),
    "kf_fp32_fma_probe": (_I32, [_P, _I64, _P, ctypes.POINTER(ctypes.c_double), _P]),
    "kf_hybrid_ffn_budget": (_I64, [_I64, _I32, _P, _P, _P]),
    "empirical_fisher_finalize": (_I32, [_P, _P, _I64, _I64, _P, _P]),
    "empirical_fisher_workspace_size": (_SZ, [_I64, _I64, _I32]),
    "empirical_fisher_accumulate": (_I32, [_P, _P, _I32, _I64, _P, _I32, _I64, _I64, _I64, _I64, _P, _I64, _P,
                                           _I64, _I32, _P, _P, _SZ, _P]),
    "activation_covariance_workspace_size": (_SZ, [_I64, _I64]),
    "activation_covariance": (_I32, [_P, _P, _I64, _I64, _P, _I32, _I64, _I64, _P, _I64, _P, _SZ, _P]),
    "activation_eig_workspace_size": (_SZ, [_I32, _I64]),
    "activation_eig": (_I32, [_P, _I32, ctypes.POINTER(SymProblem), _F, _I32, _P, _SZ, _P]),
    "activation_factors_workspace_size": (_SZ, [_I64, _I64, _I32]),
    "activation_factors": (_I32, [_P, _P, _I32, _I64, _I64, _I64, _P, _I64, _I32, _P, _I64, _P, _I64, _P, _SZ,
                                  _P]),
    "gather_rows_cols": (_I32, [_P, _P, _I32, _I64, _I64, _I64, _P, _I64, _P, _I64, _P, _I64, _P]),
    "compact_mask": (_I32, [_P, _P, _I64, _I32, _P, _P, _P]),
    "channel_errors_workspace_size": (_SZ, [_I64, _I64, _I32]),
    "channel_errors": (_I32, [_P, _P, _I32, _I64, _I64, _I64, _P, _I64, _P, _I64, _I32, _P, _I64, _P, _P, _P, _SZ,
                              _P]),
    "unwhiten_workspace_size": (_SZ, [_I64, _I64, _I32]),
    "unwhiten": (_I32, [_P, _P, _I32, _I64, _I64, _I64, _P, _I64, _P, _I64, _P, _I64, _P, _P, _I64,
                        _I32, _P, _I64, _P, _I64, _P, _SZ, _P]),
}

_lib = None


def lib() -> ctypes.CDLL:
    """Loads libkfsvd.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError("libkfsvd.so not found at %s; run __graft_entry__.build()" % LIB_PATH)
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def _check(st: int):
    if st != KF_OK:
        raise KfsvdError(st, (lib().kf_last_error() or b"").decode())


def _ptr(t) -> int:
    return 0 if t is None else int(t.data_ptr())


def _stream(stream) -> int:
    import torch
    if stream is None:
        return int(torch.cuda.current_stream().cuda_stream)
    return int(getattr(stream, "cuda_stream", stream))


def _ws(nbytes: int, workspace, device):
    import torch
    if nbytes == 0:
        return None, 0
    if workspace is not None:
        return workspace, workspace.numel() * workspace.element_size()
    return torch.empty(int(nbytes), dtype=torch.uint8, device=device), int(nbytes)


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.bfloat16:
        return KF_BF16
    if t.dtype == torch.float32:
        return KF_F32
    raise TypeError("expected bfloat16 or float32, got %s" % t.dtype)


def _ld(t) -> int:
    if t.dim() != 2 or t.stride(1) != 1:
        raise ValueError("expected a 2-D row-major tensor with unit column stride")
    return int(t.stride(0))


class Context:
    """A libkfsvd context on one device (kf_create / kf_destroy / kf_sync_status)."""

    def __init__(self, device: int = 0):
        h = ctypes.c_void_p()
        _check(lib().kf_create(int(device), ctypes.byref(h)))
        self.handle = h.value
        self.device = device

    def close(self):
        if self.handle:
            lib().kf_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def sync_status(self, stream=None) -> int:
        info = ctypes.c_int32(0)
        st = lib().kf_sync_status(self.handle, _stream(stream), ctypes.byref(info))
        if st != KF_OK:
            raise KfsvdError(st, (lib().kf_last_error() or b"").decode())
        return info.value


def kf_fp32_fma_probe(ctx: Context, iters: int, sink, stream=None) -> float:
    """Launches the FP32 FMA peak probe on ``stream``; returns the flops of the launch (the
    caller times it).  ``sink``: a float32 device tensor of 8 elements."""
    f = ctypes.c_double(0.0)
    _check(lib().kf_fp32_fma_probe(ctx.handle, int(iters), _ptr(sink), ctypes.byref(f), _stream(stream)))
    return float(f.value)


def kf_set_wait_limit(ctx: Context, limit_ns: int):
    """Limit (ns) of each tensor-core pipeline wait for later calls on ctx; 0 = the 4 s default."""
    _check(lib().kf_set_wait_limit(ctx.handle, int(limit_ns)))


def kf_hybrid_ffn_budget(budget: int, d_model: Sequence[int], n_dense: Sequence[int], with_cost: bool = False):
    """Parameters left for the low-rank factors after the dense FFN channels (host arithmetic
    in the library): max(budget - dense_cost, 0), dense_cost = sum d_model[i] n_dense[i];
    ``with_cost`` returns (left, dense_cost)."""
    k = len(d_model)
    if len(n_dense) != k:
        raise ValueError("kf_hybrid_ffn_budget: d_model and n_dense need the same length")
    a = (ctypes.c_int64 * max(k, 1))(*[int(x) for x in d_model])
    b = (ctypes.c_int64 * max(k, 1))(*[int(x) for x in n_dense])
    c = ctypes.c_int64(0)
    v = int(lib().kf_hybrid_ffn_budget(int(budget), k, ctypes.cast(a, ctypes.c_void_p),
                                       ctypes.cast(b, ctypes.c_void_p), ctypes.byref(c)))
    if v < 0:
        raise KfsvdError(KF_ERR_INVALID, (lib().kf_last_error() or b"").decode())
    return (v, int(c.value)) if with_cost else v


def kf_launch_count() -> int:
    return int(lib().kf_launch_count())


def kf_gram_side(m: int, n: int) -> int:
    return int(lib().kf_gram_side(m, n))


def kfac_accumulate_workspace_size(dtype: int, quant: int, d: int) -> int:
    return int(lib().kfac_accumulate_workspace_size(dtype, quant, d))


def kfac_accumulate(ctx: Context, act, cov_sum, quant: int = KF_QUANT_NONE, workspace=None, stream=None):
    """cov_sum (d x d float32, lower triangle) += act^T act over the rows of act."""
    n, d = act.shape
    dt = _dtype_code(act)
    ws, wsb = _ws(kfac_accumulate_workspace_size(dt, quant, d), workspace, act.device)
    _check(lib().kfac_accumulate(ctx.handle, _ptr(act), dt, n, d, _ld(act), quant, _ptr(cov_sum),
                                 _ld(cov_sum), _ptr(ws), wsb, _stream(stream)))


def fake_quant_rows(ctx: Context, rows, out, stream=None):
    """out (n_tokens x d bfloat16, contiguous) = per-token INT8 fake quantisation of rows."""
    n, d = rows.shape
    _check(lib().fake_quant_rows(ctx.handle, _ptr(rows), _dtype_code(rows), n, d, _ld(rows), _ptr(out),
                                 _stream(stream)))


def kf_finalize_covariance(ctx: Context, cov, n_tokens: int, lam: float, stream=None):
    d = cov.shape[0]
    _check(lib().kf_finalize_covariance(ctx.handle, _ptr(cov), _ld(cov), d, int(n_tokens), float(lam),
                                        _stream(stream)))


def whiten_workspace_size(m: int, n: int) -> int:
    return int(lib().whiten_workspace_size(m, n))


def whiten(ctx: Context, X, G, W, Sx, Sg, Sinv, Wt, flags: int = 0, workspace=None, stream=None):
    """Cholesky factors S_x (upper), S_g (lower), the Gram-side inverse, and W~ = S_x W S_g."""
    m, n = W.shape
    ws, wsb = _ws(whiten_workspace_size(m, n), workspace, W.device)
    _check(lib().whiten(ctx.handle, _ptr(X), _ld(X), m, _ptr(G), _ld(G), n, _ptr(W), _dtype_code(W), _ld(W),
                        int(flags), _ptr(Sx), _ld(Sx), _ptr(Sg), _ld(Sg), _ptr(Sinv), _ld(Sinv), _ptr(Wt),
                        _ld(Wt), _ptr(ws), wsb, _stream(stream)))


def factor_covariances(ctx: Context, jobs: Sequence, workspace=None, stream=None):
    """Cholesky factors (and optional inverses) of several damped covariances side by side.
    ``jobs``: tuples (A, S, Sinv or None, upper) of device tensors; S = chol_lower(A) (upper =
    False) or its transpose (upper = True), Sinv its inverse."""
    k = len(jobs)
    if k == 0:
        return
    arr = (FactorJob * k)()
    for i, (A, S, Sinv, upper) in enumerate(jobs):
        n = int(A.shape[0])
        arr[i] = FactorJob(_ptr(A), _ld(A), n, _ptr(S), _ld(S), _ptr(Sinv), 0 if Sinv is None else _ld(Sinv),
                           1 if upper else 0)
    ws, wsb = _ws(int(lib().factor_covariances_workspace_size(k, arr)), workspace, jobs[0][0].device)
    _check(lib().factor_covariances(ctx.handle, k, arr, _ptr(ws), wsb, _stream(stream)))


def kf_svd_profile_enable(ctx: Context, enable: bool = True):
    _check(lib().kf_svd_profile_enable(ctx.handle, 1 if enable else 0))


def kf_svd_profile_read(ctx: Context) -> dict:
    p = SvdProfile()
    _check(lib().kf_svd_profile_read(ctx.handle, ctypes.byref(p)))
    return {k: getattr(p, k) for k, _ in SvdProfile._fields_}


def whitened_svd_workspace_size(n_problems: int, m_max: int, n_max: int, s: int) -> int:
    return int(lib().whitened_svd_workspace_size(n_problems, m_max, n_max, s))


def whitened_svd(ctx: Context, Wts: Sequence, sigmas: Sequence, vecs: Sequence, sweeps=None,
                 tol: float = 1e-6, max_sweeps: int = 30, workspace=None, stream=None):
    """Batched spectrum of whitened weights of equal min(m, n): sigma descending, vecs the
    Gram-side singular vectors as columns.  ``sweeps`` is an int32 device tensor (one per
    problem) or None."""
    k = len(Wts)
    probs = (SvdProblem * k)()
    m_max = n_max = 0
    for i, (Wt, sg, V) in enumerate(zip(Wts, sigmas, vecs)):
        m, n = Wt.shape
        m_max, n_max = max(m_max, m), max(n_max, n)
        probs[i] = SvdProblem(_ptr(Wt), m, n, _ld(Wt), _ptr(sg), _ptr(V), _ld(V),
                              0 if sweeps is None else int(sweeps.data_ptr()) + 4 * i)
    s = min(Wts[0].shape)
    ws, wsb = _ws(whitened_svd_workspace_size(k, m_max, n_max, s), workspace, Wts[0].device)
    _check(lib().whitened_svd(ctx.handle, k, probs, float(tol), int(max_sweeps), _ptr(ws), wsb,
                              _stream(stream)))


def score_and_allocate_workspace_size(n_components: int, n_units: int) -> int:
    return int(lib().score_and_allocate_workspace_size(n_components, n_units))


def score_and_allocate(ctx: Context, sigma, seg_offset, cost, budget: int, ranks, mode: int = KF_KEY_HALF_SIGMA2,
                       fixed_rank=None, cut=None, used=None, workspace=None, stream=None):
    """Global sort-and-truncate allocation over concatenated spectra (all device tensors)."""
    n_units = int(cost.numel())
    n = int(sigma.numel()) if sigma is not None else 0
    ws, wsb = _ws(score_and_allocate_workspace_size(n, n_units), workspace, ranks.device)
    _check(lib().score_and_allocate(ctx.handle, _ptr(sigma), _ptr(seg_offset), _ptr(cost), n_units, n,
                                    int(budget), int(mode), _ptr(fixed_rank), _ptr(ranks), _ptr(cut),
                                    _ptr(used), _ptr(ws), wsb, _stream(stream)))


def score_and_allocate_weighted(ctx: Context, sigma, seg_offset, cost, budget: int, ranks,
                                mode: int = KF_KEY_ENERGY_RATIO, unit_weight=None, cut=None, used=None,
                                workspace=None, stream=None):
    """Allocation with per-unit weighted keys (UniRank: KF_KEY_ENERGY_RATIO, weight I_l)."""
    n_units = int(cost.numel())
    n = int(sigma.numel()) if sigma is not None else 0
    ws, wsb = _ws(score_and_allocate_workspace_size(n, n_units), workspace, ranks.device)
    _check(lib().score_and_allocate_weighted(ctx.handle, _ptr(sigma), _ptr(seg_offset), _ptr(cost), n_units, n,
                                             int(budget), int(mode), _ptr(unit_weight), _ptr(ranks), _ptr(cut),
                                             _ptr(used), _ptr(ws), wsb, _stream(stream)))


def score_and_allocate_keys(ctx: Context, keys, seg_offset, cost, budget: int, ranks, keep=None, cut=None, used=None,
                            workspace=None, stream=None):
    """Sort-and-truncate over given per-component keys; ``keep`` (uint8 device tensor) marks the
    kept components."""
    n_units = int(cost.numel())
    n = int(keys.numel()) if keys is not None else 0
    ws, wsb = _ws(score_and_allocate_workspace_size(n, n_units), workspace, ranks.device)
    _check(lib().score_and_allocate_keys(ctx.handle, _ptr(keys), _ptr(seg_offset), _ptr(cost), n_units, n, int(budget),
                                         _ptr(ranks), _ptr(keep), _ptr(cut), _ptr(used), _ptr(ws), wsb,
                                         _stream(stream)))


def score_and_allocate_hybrid(ctx: Context, sigma, seg_offset, cost, budget: int, ranks, alpha: float,
                              importance=None, cut=None, used=None, workspace=None, stream=None):
    """Sort-and-truncate on Swift-SVD's hybrid score beta^alpha log(e + eps*_k)^(1 - alpha), one
    key per component (``importance``: float32 device tensor of the units' beta, or None)."""
    n_units = int(cost.numel())
    n = int(sigma.numel()) if sigma is not None else 0
    ws, wsb = _ws(score_and_allocate_workspace_size(n, n_units), workspace, ranks.device)
    _check(lib().score_and_allocate_hybrid(ctx.handle, _ptr(sigma), _ptr(seg_offset), _ptr(cost), n_units, n,
                                           int(budget), _ptr(importance), float(alpha), _ptr(ranks), _ptr(cut),
                                           _ptr(used), _ptr(ws), wsb, _stream(stream)))


def empirical_fisher_finalize(ctx: Context, score_sum, n_tokens: int, keys, stream=None):
    """keys (float32) = score_sum (float64) / (2 n_tokens), rounded to float32."""
    _check(lib().empirical_fisher_finalize(ctx.handle, _ptr(score_sum), int(score_sum.numel()), int(n_tokens),
                                           _ptr(keys), _stream(stream)))


def empirical_fisher_workspace_size(m: int, n: int, r: int) -> int:
    return int(lib().empirical_fisher_workspace_size(m, n, r))


def empirical_fisher_accumulate(ctx: Context, act, grad, U, V, score_sum, workspace=None, stream=None):
    """score_sum (float64, r) += sum_t (a_t . u_i)^2 (g_t . v_i)^2 over the rows of act, grad."""
    n_tok, m = act.shape
    n = grad.shape[1]
    r = U.shape[1]
    ws, wsb = _ws(empirical_fisher_workspace_size(m, n, r), workspace, act.device)
    _check(lib().empirical_fisher_accumulate(ctx.handle, _ptr(act), _dtype_code(act), _ld(act), _ptr(grad),
                                             _dtype_code(grad), _ld(grad), n_tok, m, n, _ptr(U), _ld(U), _ptr(V),
                                             _ld(V), r, _ptr(score_sum), _ptr(ws), wsb, _stream(stream)))


def score_and_allocate_noalloc(ctx: Context, sigma, seg_offset, cost, budget: int, ranks,
                               mode: int = KF_KEY_HALF_SIGMA2, fixed_rank=None, cut=None, used=None, stream=None):
    """score_and_allocate without a workspace: for callers that cannot allocate device memory
    (its scratch is a fixed array inside the library; at most 2**20 components)."""
    n_units = int(cost.numel())
    n = int(sigma.numel()) if sigma is not None else 0
    _check(lib().score_and_allocate_noalloc(ctx.handle, _ptr(sigma), _ptr(seg_offset), _ptr(cost), n_units, n,
                                            int(budget), int(mode), _ptr(fixed_rank), _ptr(ranks), _ptr(cut),
                                            _ptr(used), _stream(stream)))


def unwhiten_workspace_size(m: int, n: int, r: int) -> int:
    return int(lib().unwhiten_workspace_size(m, n, r))


def unwhiten(ctx: Context, W, Sx, Sg, Sinv, sigma, vecs, r: int, U, V, workspace=None, stream=None):
    """Rank-r factors U (m x r), V (r x n) with W ~= U V in the original space.  Only the
    Gram-side factor is read (Sg when n <= m, else Sx); the other may be None."""
    m, n = W.shape
    ws, wsb = _ws(unwhiten_workspace_size(m, n, r), workspace, W.device)
    _check(lib().unwhiten(ctx.handle, _ptr(W), _dtype_code(W), _ld(W), m, n, _ptr(Sx),
                          0 if Sx is None else _ld(Sx), _ptr(Sg), 0 if Sg is None else _ld(Sg),
                          _ptr(Sinv), _ld(Sinv), _ptr(sigma), _ptr(vecs), _ld(vecs), int(r), _ptr(U),
                          _ld(U) if r > 0 else max(r, 1), _ptr(V), _ld(V), _ptr(ws), wsb, _stream(stream)))


# ------------------------------------------------- Swift-SVD activation-only route
def activation_covariance(ctx: Context, X, W, C, workspace=None, stream=None):
    """C (n x n) = W^T X W: the covariance of the layer output y = a W from the activation
    second moment X (m x m, full symmetric)."""
    m, n = W.shape
    ws, wsb = _ws(int(lib().activation_covariance_workspace_size(m, n)), workspace, W.device)
    _check(lib().activation_covariance(ctx.handle, _ptr(X), _ld(X), m, _ptr(W), _dtype_code(W), _ld(W), n,
                                       _ptr(C), _ld(C), _ptr(ws), wsb, _stream(stream)))


def activation_eig(ctx: Context, Cs: Sequence, sigmas: Sequence, vecs: Sequence, sweeps=None,
                   tol: float = 1e-6, max_sweeps: int = 30, workspace=None, stream=None):
    """Batched eigenpairs of symmetric C of equal size: sigma = sqrt(max(lambda, 0))
    descending, vecs the eigenvectors as columns."""
    k = len(Cs)
    probs = (SymProblem * k)()
    for i, (C, sg, V) in enumerate(zip(Cs, sigmas, vecs)):
        n = C.shape[0]
        probs[i] = SymProblem(_ptr(C), n, _ld(C), _ptr(sg), _ptr(V), _ld(V),
                              0 if sweeps is None else int(sweeps.data_ptr()) + 4 * i)
    n0 = Cs[0].shape[0]
    ws, wsb = _ws(int(lib().activation_eig_workspace_size(k, n0)), workspace, Cs[0].device)
    _check(lib().activation_eig(ctx.handle, k, probs, float(tol), int(max_sweeps), _ptr(ws), wsb, _stream(stream)))


def activation_factors(ctx: Context, W, vecs, r: int, U, V, workspace=None, stream=None):
    """U = W V_r (m x r), V = V_r^T (r x n) for the first r eigenvector columns V_r of vecs."""
    m, n = W.shape
    ws, wsb = _ws(int(lib().activation_factors_workspace_size(m, n, r)), workspace, W.device)
    _check(lib().activation_factors(ctx.handle, _ptr(W), _dtype_code(W), _ld(W), m, n, _ptr(vecs), _ld(vecs),
                                    int(r), _ptr(U), _ld(U) if r > 0 else max(r, 1), _ptr(V), _ld(V), _ptr(ws),
                                    wsb, _stream(stream)))


# ------------------------------------------------- LASER hybrid FFN channel selection
def channel_errors(ctx: Context, W, U, V, X, err_sum, keys=None, workspace=None, stream=None):
    """err_sum (float64, n) += per-channel errors d_j^T X d_j of W - U V; keys (float32, n) =
    float(err_sum) afterwards if given.  U (m x r) / V (r x n) may be None for r = 0."""
    m, n = W.shape
    r = 0 if U is None else int(U.shape[1])
    ws, wsb = _ws(int(lib().channel_errors_workspace_size(m, n, r)), workspace, W.device)
    _check(lib().channel_errors(ctx.handle, _ptr(W), _dtype_code(W), _ld(W), m, n, _ptr(U),
                                _ld(U) if r > 0 else 1, _ptr(V), _ld(V) if r > 0 else n, r, _ptr(X), _ld(X),
                                _ptr(err_sum), _ptr(keys), _ptr(ws), wsb, _stream(stream)))


# ------------------------------------------------------------- index plumbing
def gather_rows_cols(ctx: Context, src, row_idx=None, col_idx=None, out=None, stream=None):
    """out = src[row_idx][:, col_idx] (either index may be None: all rows / columns), by the
    library's gather kernel; int64 device indices."""
    import torch
    R, C = src.shape
    rows = R if row_idx is None else int(row_idx.numel())
    cols = C if col_idx is None else int(col_idx.numel())
    if out is None:
        out = torch.empty((rows, max(cols, 1)), dtype=src.dtype, device=src.device)[:, :cols]
    _check(lib().gather_rows_cols(ctx.handle, _ptr(src), _dtype_code(src), _ld(src), R, C, _ptr(row_idx), rows,
                                  _ptr(col_idx), cols, _ptr(out), _ld(out) if cols > 0 else 1, _stream(stream)))
    return out


def compact_mask(ctx: Context, mask, want: int = 1, stream=None):
    """Increasing positions where mask (uint8) is nonzero (want=1) or zero (want=0), as an
    int64 device tensor (one host read of the count)."""
    import torch
    n = int(mask.numel())
    idx = torch.empty(max(n, 1), dtype=torch.int64, device=mask.device)
    cnt = torch.zeros(1, dtype=torch.int64, device=mask.device)
    _check(lib().compact_mask(ctx.handle, _ptr(mask), n, int(want), _ptr(idx), _ptr(cnt), _stream(stream)))
    return idx[:int(cnt.item())]
