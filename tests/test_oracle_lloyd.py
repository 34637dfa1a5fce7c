"""Pins of the Lloyd-Max codebook oracle (oracle/lloyd.py)."""
import numpy as np

import oracle
from oracle import lloyd as L


def test_a_equal_one_is_round_to_nearest():
    rng = np.random.default_rng(1)
    u = rng.uniform(0, 3, 100000)
    u = u[np.abs(u - np.floor(u) - 0.5) > 1e-9]          # away from exact ties
    assert np.array_equal(L.codes_from_u(u, 1.0), np.clip(np.rint(u), 0, 3).astype(np.uint8))


def test_codes_are_nearest_levels():
    rng = np.random.default_rng(2)
    for a in (0.6, 1.0, 1.3):
        u = rng.uniform(0, 3, 5000)
        lv = L.levels(a)
        brute = np.argmin(np.abs(u[:, None] - lv[None, :]), axis=1)
        assert np.array_equal(L.codes_from_u(u, a), brute)


def test_lloyd_on_uniform_samples_gives_the_uniform_grid():
    # u uniform on [0, 3]: the folded u' is uniform on [0, 1.5]; the cell of a
    # is [a/2, 1.5] with mean a/4 + 3/4, whose fixed point is a = 1
    u = np.linspace(0, 3, 300001)
    assert abs(L.fit_a(u, 0.5) - 1.0) < 1e-5


def test_lloyd_fixed_point_for_a_two_point_distribution():
    # u' in {0, 1.2} (equal mass): from any start in (0, 2.4) the cell of a
    # holds exactly the 1.2 samples, so a = 1.2
    u = np.array([0.0, 1.2, 1.8, 3.0] * 100)
    assert abs(L.fit_a(u, 1.0) - 1.2) < 1e-12


def test_lloyd_decreases_the_quantisation_error():
    rng = np.random.default_rng(3)
    u = np.clip(rng.normal(1.5, 0.6, 20000), 0, 3)        # concentrated in the middle
    a = L.fit_a(u)
    err = lambda aa: np.mean((u - L.levels(aa)[L.codes_from_u(u, aa)]) ** 2)  # noqa: E731
    assert a > 1.0 and err(a) < err(1.0)
    for da in (-0.02, 0.02):                              # a local minimum of the error
        assert err(a) <= err(a + da) + 1e-12


def test_dequantize_with_a_one_matches_the_c_oracle():
    orc = oracle.get()
    rng = np.random.default_rng(4)
    y = rng.standard_normal(128) * 2
    codes, s16, z16 = orc.quantize_vec(y, 32, 0.95)[:3]
    ref = orc.dequantize_vec(codes, s16, z16, 32)
    mine = L.dequantize(codes, L._f16(s16), L._f16(z16), 1.0, 32)
    assert np.allclose(mine, ref, rtol=0, atol=0)
