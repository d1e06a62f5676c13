"""The C ABI library loads on a host without a GPU, exports every declared symbol, and
rejects bad arguments synchronously (no compute calls here)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kfsvd.h")


def declared_symbols():
    txt = open(HEADER).read()
    return sorted(set(re.findall(r"^KF_API [^(]*?\b([a-z_][a-z_0-9]*)\(", txt, flags=re.M)))


def test_header_declares_the_five_steps():
    syms = declared_symbols()
    for s in ("kfac_accumulate", "whiten", "whitened_svd", "score_and_allocate", "unwhiten"):
        assert s in syms


def test_library_exports_every_declared_symbol():
    from vlm_compression_fac_b300 import kfsvd as K
    L = K.lib()
    missing = [s for s in declared_symbols() if not hasattr(L, s)]
    assert not missing, missing
    assert sorted(K.EXPORTED) == declared_symbols()


def test_library_has_no_driver_link_dependency():
    # the .so must load without libcuda (driver entry points are resolved at run time)
    from vlm_compression_fac_b300 import kfsvd as K
    out = os.popen("ldd %s" % K.LIB_PATH).read()
    assert "libcuda.so" not in out and "libtorch" not in out


def test_workspace_queries_are_host_only():
    from vlm_compression_fac_b300 import kfsvd as K
    assert K.kfac_accumulate_workspace_size(K.KF_BF16, K.KF_QUANT_NONE, 4096) == 0
    assert K.kfac_accumulate_workspace_size(K.KF_F32, K.KF_QUANT_NONE, 256) >= 2 * 8192 * 256 * 2
    assert K.whiten_workspace_size(4096, 11008) >= 4096 * 11008 * 4
    assert K.whitened_svd_workspace_size(7, 11008, 11008, 4096) >= 7 * 2 * 4096 * 4096 * 4
    assert K.score_and_allocate_workspace_size(1 << 20, 7) >= 2 * 8 * (1 << 20)  # two key buffers
    assert K.unwhiten_workspace_size(4096, 4096, 0) == 0
    assert K.kf_gram_side(4096, 4096) == K.KF_SIDE_RIGHT
    assert K.kf_gram_side(4096, 11008) == K.KF_SIDE_LEFT
    assert K.kf_gram_side(11008, 4096) == K.KF_SIDE_RIGHT


def test_invalid_arguments_fail_before_any_launch():
    from vlm_compression_fac_b300 import kfsvd as K
    L = K.lib()
    st = L.kfac_accumulate(None, None, 0, 10, 8, 8, 0, None, 8, None, 0, None)
    assert st == K.KF_ERR_INVALID
    assert b"null context" in L.kf_last_error()
    st = L.score_and_allocate(None, None, None, None, 1, 0, 0, 0, None, None, None, None, None, 0, None)
    assert st == K.KF_ERR_INVALID
    assert L.kf_sync_status(None, None, None) == K.KF_ERR_INVALID
    h = ctypes.c_void_p()
    st = L.kf_create(0, ctypes.byref(h))
    if st != K.KF_OK:          # no GPU on this host: a clean error, no crash
        assert st in (K.KF_ERR_CUDA, K.KF_ERR_UNSUPPORTED, K.KF_ERR_INVALID)
    else:
        L.kf_destroy(h)


def test_every_compute_call_rejects_a_null_context():
    """Each entry point's argument check runs on the host before any CUDA call: with a null
    context every compute call returns KF_ERR_INVALID and names itself in kf_last_error."""
    from vlm_compression_fac_b300 import kfsvd as K
    L = K.lib()
    calls = {
        "fake_quant_rows": (None, None, 0, 4, 8, 8, None, None),
        "whiten": (None,) + (None, 8, 8, None, 8, 8, None, 0, 8, 0, None, 8, None, 8, None, 8, None, 8, None, 0, None),
        "whitened_svd": (None, 1, None, 1e-6, 30, None, 0, None),
        "score_and_allocate_weighted": (None, None, None, None, 1, 0, 0, 3, None, None, None, None, None, 0, None),
        "score_and_allocate_keys": (None, None, None, None, 1, 0, 0, None, None, None, None, None, 0, None),
        "empirical_fisher_accumulate": (None, None, 0, 8, None, 0, 8, 4, 8, 8, None, 8, None, 8, 8, None, None, 0,
                                        None),
        "unwhiten": (None, None, 0, 8, 8, 8, None, 8, None, 8, None, 8, None, None, 8, 1, None, 1, None, 8, None, 0,
                     None),
        "activation_covariance": (None, None, 8, 8, None, 0, 8, 8, None, 8, None, 0, None),
        "activation_eig": (None, 1, None, 1e-6, 30, None, 0, None),
        "activation_factors": (None, None, 0, 8, 8, 8, None, 8, 1, None, 1, None, 8, None, 0, None),
        "channel_errors": (None, None, 0, 8, 8, 8, None, 1, None, 8, 1, None, 8, None, None, None, 0, None),
        "gather_rows_cols": (None, None, 0, 8, 8, 8, None, 1, None, 1, None, 1, None),
        "compact_mask": (None, None, 4, 1, None, None, None),
        "empirical_fisher_finalize": (None, None, 4, 10, None, None),
        "score_and_allocate_hybrid": (None, None, None, None, 1, 0, 0, None, 0.5, None, None, None, None, 0, None),
        "kf_set_wait_limit": (None, 1000),
        "factor_covariances": (None, 1, None, None, 0, None),
    }
    for name, args in calls.items():
        st = getattr(L, name)(*args)
        assert st == K.KF_ERR_INVALID, name
        msg = L.kf_last_error()
        assert name.encode() in msg and b"null context" in msg, (name, msg)


def test_hybrid_allocation_and_budget_reject_bad_arguments_on_the_host():
    """score_and_allocate_hybrid checks alpha in [0, 1] before any launch; the hybrid FFN budget
    is host arithmetic in the library (equal to the oracle's statement of it)."""
    import oracle as O
    from vlm_compression_fac_b300 import kfsvd as K
    L = K.lib()
    h = ctypes.c_void_p(1)   # never dereferenced: the alpha check comes first
    st = L.score_and_allocate_hybrid(h, None, None, None, 1, 0, 0, None, 1.5, None, None, None, None, 0, None)
    assert st == K.KF_ERR_INVALID and b"alpha" in L.kf_last_error()
    for budget, dm, nd in ((1000, [64, 64], [3, 3]), (100, [64, 64], [3, 3]), (7, [], []), (10 ** 12, [4096] * 4,
                                                                                            [1000, 2000, 0, 7])):
        assert K.kf_hybrid_ffn_budget(budget, dm, nd) == O.hybrid_ffn_budget(budget, dm, nd)
    with pytest.raises(K.KfsvdError):
        K.kf_hybrid_ffn_budget(10, [64], [-1])
