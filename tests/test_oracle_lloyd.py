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


def test_dequantised_values_reproduce_the_nearest_level():
    # for a != 1: u -> code -> value must give back the level of R26 nearest
    # to u (unit scale, zero offset), written out here as {0, a, 3 - a, 3}
    rng = np.random.default_rng(6)
    for a in (0.6, 1.3):
        u = rng.uniform(0, 3, 128)
        v = L.dequantize(L.codes_from_u(u, a), np.ones(4), np.zeros(4), a, 32)
        lv = np.array([0.0, a, 3.0 - a, 3.0])
        assert np.allclose(v, lv[np.argmin(np.abs(u[:, None] - lv[None, :]), axis=1)], rtol=0, atol=1e-15)


def test_dequantize_with_a_one_matches_the_c_oracle():
    orc = oracle.get()
    rng = np.random.default_rng(4)
    y = rng.standard_normal(128) * 2
    codes, s16, z16 = orc.quantize_vec(y, 32, 0.95)[:3]
    ref = orc.dequantize_vec(codes, s16, z16, 32)
    mine = L.dequantize(codes, L._f16(s16), L._f16(z16), 1.0, 32)
    assert np.allclose(mine, ref, rtol=0, atol=0)


def test_decode_with_a_one_is_the_c_oracle_decode():
    """With a = 1 the levels are the uniform ones, so the variant's decode
    (stored codes dequantised with the levels, mapped back by R^T) equals
    the C oracle's plain decode on the same pool."""
    from bit_kv_cache_evict_gb300 import synth as S
    orc = oracle.get()
    w = S.Workload(31, "lloyd_pin", batch=2, hq=4, hk=2)
    shape = oracle.Shape(128, 32, 64, 256, 64, 4, 2)
    hist = np.array([130, 70], np.int32)
    rc, table, npages, nbytes = orc.pool_layout(shape, hist)
    assert rc == 0
    rng = S.rng_for(w, 2)
    prof = S.channel_profile(w)
    src = np.concatenate([S.kv_tokens(w, int(h), rng, prof) for h in hist])
    seq = np.concatenate([np.full(h, b, np.int32) for b, h in enumerate(hist)])
    pos = np.concatenate([np.arange(h, dtype=np.int32) for h in hist])
    U = S.rotation_U(w).astype(np.float64)
    pool = np.zeros(nbytes, np.uint8)
    orc.evict(shape, src, seq, pos, U, S.clip_ratios(w), pool, table, table.shape[1])
    bkv = S.kv_tokens(w, 2 * 320, rng, prof).reshape(2, 320, 2, 2, 128)
    blen = np.array([320, 7], np.int32)
    q = S.queries(w, rng, 2)
    ref = orc.decode(shape, q, bkv, blen, pool, table, table.shape[1], hist, U, 0.09)
    got = L.decode(q, bkv, blen, pool, table, hist, U, orc.build_R, np.ones((2, 2)), 0.09, 32)
    assert np.abs(got - ref).max() < 1e-12
