"""Pins of the offline-calibration oracle (oracle/calibrate.py).

Each check compares the oracle with something fixed independently of its
code: a covariance built from a known eigenbasis, attention cases with a
closed form, and the defining eigen-equations.
"""
import numpy as np
import pytest

from oracle import calibrate as C

D = 128


def _orthogonal(seed: int) -> np.ndarray:
    rng = np.random.default_rng(seed)
    q, r = np.linalg.qr(rng.standard_normal((D, D)))
    return q * np.sign(np.diag(r))[None, :]


def test_known_eigenbasis_is_recovered_in_order_with_signs():
    Q = _orthogonal(11)
    lam = np.exp(-np.arange(D) / 20.0) * 5.0
    perm = np.random.default_rng(3).permutation(D)      # eigenvalues in scrambled column order
    Cm = (Q[:, perm] * lam[perm]) @ Q[:, perm].T
    U, w = C.rotation_from_covariance(Cm)
    assert np.allclose(w, lam, rtol=1e-12, atol=1e-12)
    # column j is +-Q[:, j] (lam decreasing), with its largest-magnitude entry positive
    dots = np.einsum("ij,ij->j", U, Q)
    assert np.allclose(np.abs(dots), 1.0, atol=1e-10)
    for j in range(D):
        i = int(np.argmax(np.abs(U[:, j])))
        assert U[i, j] > 0
        assert np.allclose(U[:, j], np.sign(Q[i, j]) * Q[:, j], atol=1e-10)


def test_eigen_equations_and_orthogonality():
    rng = np.random.default_rng(5)
    X = rng.standard_normal((300, D)) * np.exp(-np.arange(D) / 40.0)
    Cm = X.T @ X / 300
    U, w = C.rotation_from_covariance(Cm)
    assert np.abs(U.T @ U - np.eye(D)).max() < 1e-12
    assert np.abs(Cm @ U - U * w).max() < 1e-10 * w[0]
    assert np.all(np.diff(w) <= 0)


def test_query_covariance_of_a_constructed_sample_set():
    # d samples x_n = sqrt(d * lam_n) Q[:, n] have mean outer product Q diag(lam) Q^T
    Q = _orthogonal(7)
    lam = 1.0 + np.arange(D)[::-1] * 0.1
    x = (np.sqrt(D * lam)[:, None] * Q.T)                # [n=d][d]
    Cm = C.query_covariance(x[:, None, :], 1)[0]
    assert np.allclose(Cm, (Q * lam) @ Q.T, atol=1e-11)


def test_query_covariance_groups_query_heads_by_kv_head():
    rng = np.random.default_rng(2)
    q = rng.standard_normal((5, 4, D))                   # 4 query heads, 2 KV heads: heads {0,1} -> 0, {2,3} -> 1
    Cm = C.query_covariance(q, 2)
    brute = np.zeros((D, D))
    for n in range(5):
        for h in (2, 3):
            brute += np.outer(q[n, h], q[n, h])
    assert np.allclose(Cm[1], brute / 10, atol=1e-12)


def test_attention_outputs_closed_forms():
    rng = np.random.default_rng(9)
    t = 40
    v = rng.standard_normal((t, 1, D))
    # identical keys: uniform weights, the output is the mean value
    k = np.repeat(rng.standard_normal((1, 1, D)), t, axis=0)
    q = rng.standard_normal((3, 2, D))
    o = C.attention_outputs(q, k, v, 0.1)
    assert np.allclose(o, np.broadcast_to(v[:, 0, :].mean(axis=0), o.shape), atol=1e-12)
    # one key along the query with a huge logit: the output is that token's value
    k2 = rng.standard_normal((t, 1, D)) * 1e-3
    k2[17, 0] = q[0, 0] * 50.0
    o2 = C.attention_outputs(q[:1, :1], k2, v, 1.0)
    assert np.allclose(o2[0, 0], v[17, 0], atol=1e-12)


def test_value_covariance_is_the_output_covariance():
    rng = np.random.default_rng(4)
    o = rng.standard_normal((6, 2, D))
    assert np.allclose(C.value_covariance(o, 1)[0], sum(np.outer(x, x) for x in o.reshape(12, D)) / 12)


def test_calibrate_end_to_end_on_a_small_case():
    from bit_kv_cache_evict_gb300 import synth as S
    qb, kvb = S.calibration_inputs(3, 64, 96, 4, 1)
    q = S.bf16_to_f32(qb).astype(np.float64)
    kv = S.bf16_to_f32(kvb).astype(np.float64)
    U, lam = C.calibrate(q, kv, 1 / np.sqrt(D))
    ck = C.query_covariance(q, 1)[0]
    assert np.abs(ck @ U[0, 0] - U[0, 0] * lam[0, 0]).max() < 1e-9 * lam[0, 0, 0]
    for w in range(2):
        assert np.abs(U[0, w].T @ U[0, w] - np.eye(D)).max() < 1e-12


def _minmax_mse(Y: np.ndarray, g: int) -> float:
    """Textbook min-max asymmetric INT2 (fp16 scale/zero, round half to even)
    computed with numpy alone."""
    err = 0.0
    for y in Y:
        for k in range(0, y.size, g):
            v = y[k:k + g]
            lo, hi = v.min(), v.max()
            s = float(np.float16((hi - lo) / 3))
            z = float(np.float16(lo))
            codes = np.zeros(g) if s == 0 else np.clip(np.rint((v - z) / s), 0, 3)
            err += float(((v - (s * codes + z)) ** 2).sum())
    return err / Y.size


def test_clip_search_without_clipping_is_textbook_minmax():
    from oracle import get
    rng = np.random.default_rng(12)
    kv = rng.standard_normal((20, 1, 2, D))
    U = np.stack([_orthogonal(1), _orthogonal(2)])[None]
    clip, mse = C.clip_search(kv, U, [1.0])
    assert clip[0, 0] == 1.0 and clip[0, 1] == 1.0
    Y = kv[:, 0, 0, :] @ get().build_R(U[0, 0])
    assert np.isclose(mse[0, 0, 0], _minmax_mse(Y, 32), rtol=1e-12)


def test_clip_search_prefers_clipping_a_lone_outlier():
    # after the rotation every group holds N(0, 1)-like values; add one large
    # value per group in the rotated domain through U = identity-like setup
    from oracle import get
    rng = np.random.default_rng(13)
    R = get().build_R(np.eye(D))
    Y = rng.standard_normal((40, D))
    Y[:, ::32] = 12.0                                    # one value per 32-position group far out
    kv = (Y @ R.T)[:, None, None, :].repeat(2, axis=2)   # x with x . R = Y
    clip, mse = C.clip_search(kv, np.eye(D)[None, None].repeat(2, axis=1), [0.3, 0.6, 1.0])
    assert clip[0, 0] < 1.0
    assert mse[0, 0, 2] > mse[0, 0, list([0.3, 0.6, 1.0]).index(clip[0, 0])]


def test_two_token_attention_is_a_logistic_mix():
    # two keys: the output is v0 + sigmoid(sm (q.k1 - q.k0)) (v1 - v0)
    rng = np.random.default_rng(21)
    q = rng.standard_normal((3, 1, D))
    k = rng.standard_normal((2, 1, D))
    v = rng.standard_normal((2, 1, D))
    sm = 0.37
    o = C.attention_outputs(q, k, v, sm)
    for n in range(3):
        lam = 1.0 / (1.0 + np.exp(-sm * (q[n, 0] @ k[1, 0] - q[n, 0] @ k[0, 0])))
        assert np.allclose(o[n, 0], v[0, 0] + lam * (v[1, 0] - v[0, 0]), atol=1e-12)


def test_value_rotation_of_uniform_attention_is_the_mean_value():
    # identical keys: every output is the mean value m, so C_V = m m^T and the
    # first column of U_V is m / |m| (sign convention: largest entry positive)
    # with eigenvalue |m|^2
    rng = np.random.default_rng(22)
    n_t = 50
    kv = np.zeros((n_t, 1, 2, D))
    kv[:, 0, 0, :] = rng.standard_normal(D)             # the same key for every token
    kv[:, 0, 1, :] = rng.standard_normal((n_t, D)) + 0.5
    q = rng.standard_normal((7, 2, D))
    U, lam = C.calibrate(q, kv, 0.2)
    m = kv[:, 0, 1, :].mean(axis=0)
    u0 = m / np.linalg.norm(m)
    u0 = u0 if u0[np.argmax(np.abs(u0))] > 0 else -u0
    assert np.allclose(U[0, 1, :, 0], u0, atol=1e-9)
    assert np.isclose(lam[0, 1, 0], m @ m, rtol=1e-10)
