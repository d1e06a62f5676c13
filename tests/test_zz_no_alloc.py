"""score_and_allocate_noalloc: the allocation entry point for callers that cannot allocate
device memory (a framework that owns all GPU memory, or code that must not trigger an
allocation mid-job).  Its results must equal those of score_and_allocate, which uses a
caller workspace, on consecutive calls that share the library's fixed scratch array.

Kept in its own file so that pytest collects it after every other test.
"""
import ctypes

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def _problem(seed, n_units, max_len):
    r = np.random.default_rng(seed)
    sig, costs = [], []
    for _ in range(n_units):
        m, n = int(r.integers(8, max_len + 8)), int(r.integers(8, max_len + 8))
        sig.append(np.sort(r.gamma(1.0, 1.0, size=min(m, n)))[::-1].astype(np.float32))
        costs.append(m + n)
    budget = int(0.4 * sum(len(s) * c for s, c in zip(sig, costs)))
    dev = "cuda"
    return (torch.from_numpy(np.concatenate(sig)).to(dev),
            torch.tensor([0] + list(np.cumsum([len(s) for s in sig])), dtype=torch.int64, device=dev),
            torch.tensor(costs, dtype=torch.int64, device=dev), budget, n_units)


def _outputs(n_units):
    return (torch.full((n_units,), -1, dtype=torch.int32, device="cuda"),
            torch.zeros(2, dtype=torch.float32, device="cuda"),
            torch.full((1,), -1, dtype=torch.int64, device="cuda"))


def test_noalloc_matches_workspace_entry_point_on_consecutive_calls():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from vlm_compression_fac_b300 import kfsvd as K
    L = K.lib()
    ctx = K.Context(0)
    stream = torch.cuda.current_stream().cuda_stream
    # a large call first, then a smaller one: the second must not see the first's leftovers
    for seed, nu, ml, mode in ((1, 300, 3000, K.KF_KEY_HALF_SIGMA2), (2, 40, 500, K.KF_KEY_PER_PARAM)):
        sig, off, cost, budget, n_units = _problem(seed, nu, ml)
        r_ws, c_ws, u_ws = _outputs(n_units)
        K.score_and_allocate(ctx, sig, off, cost, budget, r_ws, mode=mode, cut=c_ws, used=u_ws)
        r_na, c_na, u_na = _outputs(n_units)
        st = L.score_and_allocate_noalloc(ctx.handle, sig.data_ptr(), off.data_ptr(), cost.data_ptr(), n_units,
                                          sig.numel(), budget, mode, None, r_na.data_ptr(), c_na.data_ptr(),
                                          u_na.data_ptr(), ctypes.c_void_p(stream))
        assert st == K.KF_OK, L.kf_last_error()
        ctx.sync_status()
        assert torch.equal(r_ws, r_na)                       # integer results: bit-exact
        assert torch.equal(u_ws, u_na)
        assert np.array_equal(c_ws.cpu().numpy().view(np.uint32), c_na.cpu().numpy().view(np.uint32))
        assert int(r_na.min()) >= 0 and int(u_na.item()) <= budget
    # beyond the stated maximum: rejected on the host, nothing launched
    st = L.score_and_allocate_noalloc(ctx.handle, sig.data_ptr(), off.data_ptr(), cost.data_ptr(), n_units,
                                      (1 << 20) + 1, budget, K.KF_KEY_HALF_SIGMA2, None, r_na.data_ptr(), None, None,
                                      ctypes.c_void_p(stream))
    assert st == K.KF_ERR_UNSUPPORTED and b"1048576" in L.kf_last_error()
    ctx.close()
