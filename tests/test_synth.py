"""Seeded input generator: determinism, slicing consistency, distributions (CPU)."""
import numpy as np

from synth import philox, recipes


def test_normal_moments_and_determinism():
    e = np.arange(1 << 18, dtype=np.uint64)
    z1 = philox.standard_normal(e, 99)
    z2 = philox.standard_normal(e, 99)
    np.testing.assert_array_equal(z1, z2)
    assert abs(float(z1.mean())) < 0.01 and abs(float(z1.std()) - 1.0) < 0.01
    assert np.abs(z1).max() <= 6.0
    z3 = philox.standard_normal(e, 100)
    assert abs(float(np.corrcoef(z1, z3)[0, 1])) < 0.01


def test_irwin_hall_values_are_exact_float32_grid():
    z = philox.standard_normal(np.arange(4096, dtype=np.uint64), 5)
    k = z.astype(np.float64) * 65536.0
    np.testing.assert_array_equal(k, np.round(k))


def test_stream_slicing_is_consistent():
    wl = recipes.mini_block()
    site = wl.sites["down_in"]
    full = recipes.gen_stream(wl, site, 0, 64)
    part = recipes.gen_stream(wl, site, 17, 40, cols=[3, 100, 703])
    np.testing.assert_array_equal(full[17:40][:, [3, 100, 703]], part)


def test_bf16_rounding_is_nearest_even():
    x = np.array([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -1.0 - 2 ** -8, 1.0 + 2 ** -8 + 2 ** -20],
                 dtype=np.float32)
    got = philox.bf16_bits_to_f32(philox.f32_to_bf16_bits(x))
    np.testing.assert_array_equal(got, np.array([1.0, 1.0 + 2 ** -6, -1.0, 1.0 + 2 ** -7],
                                                dtype=np.float32))


def test_workload_shapes_and_budgets():
    wl = recipes.llama7b_block()
    assert len(wl.units) == 7 and wl.n_tokens == 131072
    assert wl.budget == 101187584
    assert sorted({(u.m, u.n) for u in wl.units}) == [(4096, 4096), (4096, 11008), (11008, 4096)]
    assert recipes.llama70b_block().budget == 256691404
    out = recipes.outlier_channels(wl, wl.sites["down_in"])
    assert len(out) == 110 and len(set(out.tolist())) == 110
    std = recipes.site_std(wl, wl.sites["attn_in"])
    assert int(np.sum(std == 20.0)) == 41 and int(np.sum(std == 1.0)) == 4096 - 41


def test_powerlaw_spectrum():
    wl = recipes.single_linear()
    A = recipes.gen_stream(wl, wl.sites["in"], 0, 2048)
    v = A.astype(np.float64).var(axis=0)
    i = np.arange(1, 257)
    assert np.all(np.abs(v * i - 1.0) < 0.2)
